// Tree attention (K4): all tree tokens attend, in one pass, to the KV cache and
// to their own ancestors in the candidate tree.
//
// wiblog.cn "Medusa multi-head speculative decoding", section "Tree attention":
// inside one path the usual causal mask holds, different paths must not see
// each other, so each token attends only to the tokens on its prefix path; the
// tree is fixed, so the mask is prepared once and cached.  Ultralytics
// glossary "Medusa Heads", section "Tree attention and accepting tokens": all
// candidate tokens enter one forward pass and the mask lets each token see
// only its ancestors.
//
// bf16 path: split-KV ("flash-decoding") over the cache plus one extra split
// for the tree segment, where the cached ancestor bitmask masks the scores.
// One CTA owns a tile of up to 128 query rows of one KV head: a query row is
// (node, query head of this KV head's group), so the heads that share a KV
// head share every K/V tile load.  K/V tiles are staged in shared memory by
// cp.async (double buffered), QK^T and PV run on mma.sync bf16 tensor-core
// tiles with fp32 accumulation and an fp32 online softmax.  A second kernel
// merges the splits.  fp32 path: an exact scalar kernel (small shapes).
#include <algorithm>

#include "tree.cuh"

using namespace medusa;

namespace {

constexpr int KB = 64;  // keys per smem tile

struct AttnPlan {
  int G, R, n_qt, rows_per_tile, nwarps, n_splits, chunk, n_parts, R_pad;
};

AttnPlan plan_attn(int T, int B, int Hq, int Hkv, int Lmax, int hint) {
  AttnPlan p{};
  p.G = Hq / Hkv;
  p.R = T * p.G;
  p.n_qt = cdiv(p.R, 128);
  p.rows_per_tile = cdiv(cdiv(p.R, p.n_qt), 16) * 16;
  p.nwarps = p.rows_per_tile / 16;
  p.R_pad = p.n_qt * p.rows_per_tile;
  const int L = hint > 0 ? std::min(hint, Lmax) : Lmax;
  const int base = B * Hkv * p.n_qt;
  const int target = 2 * 148;
  int ns = std::max(1, (target + base / 2) / base);
  ns = std::max(ns, cdiv(std::max(L, 1), 1024));
  ns = std::min(ns, std::max(1, cdiv(std::max(L, 1), KB)));
  p.chunk = cdiv(cdiv(std::max(L, 1), ns), KB) * KB;
  p.n_splits = cdiv(std::max(L, 1), p.chunk);
  p.n_parts = p.n_splits + 1;
  return p;
}

size_t attn_ws_bytes(const AttnPlan& p, int B, int Hkv, int D) {
  const size_t nrow = static_cast<size_t>(B) * Hkv * p.n_parts * p.R_pad;
  return align_up(nrow * D * 4, 256) + align_up(nrow * 8, 256);
}

__device__ inline uint32_t ld_u32(const __nv_bfloat16* p) { return *reinterpret_cast<const uint32_t*>(p); }

__device__ inline void cp_async16(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0));
}
__device__ inline void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N> __device__ inline void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

__device__ inline void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ inline void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ inline void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
               : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
               : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ inline uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Swizzled smem tile [KB keys][D]: 16-byte chunk c of key row j sits at c ^ (j & 7).
template <int D>
__device__ inline uint32_t tile_addr(uint32_t base, int key, int chunk) {
  return base + key * (D * 2) + ((chunk ^ (key & 7)) << 4);
}

template <int D>
__global__ void __launch_bounds__(256) tree_attn_bf16_kernel(
    medusa_tree_dev tr, const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k_new,
    const __nv_bfloat16* __restrict__ v_new, const __nv_bfloat16* __restrict__ k_cache,
    const __nv_bfloat16* __restrict__ v_cache, const int32_t* __restrict__ kv_len, int Hq, int Hkv, int Lmax,
    AttnPlan p, float scale_log2, float* __restrict__ o_part, float2* __restrict__ ml_part) {
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int NCH = D / 8;  // 16-byte chunks per row
  const int part = blockIdx.x, qt = blockIdx.y, zb = blockIdx.z;
  const int b = zb / Hkv, g = zb % Hkv;
  const int T = tr.T, G = p.G, R = p.R;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, tq = lane & 3;
  const int row0 = qt * p.rows_per_tile + warp * 16;
  const bool is_tree = part == p.n_splits;
  const int L = min(max(kv_len[b], 0), Lmax);

  const uint32_t sK = smem_u32(smem);
  const uint32_t sV = sK + 2 * KB * D * 2;

  // query fragments (A operand) for this warp's 16 rows
  const int ra = row0 + gq, rb = row0 + gq + 8;
  const int node_a = ra < R ? ra / G : -1, node_b = rb < R ? rb / G : -1;
  const __nv_bfloat16* qa_ptr = node_a >= 0 ? q + ((static_cast<size_t>(b) * T + node_a) * Hq + g * G + ra % G) * D : nullptr;
  const __nv_bfloat16* qb_ptr = node_b >= 0 ? q + ((static_cast<size_t>(b) * T + node_b) * Hq + g * G + rb % G) * D : nullptr;
  uint32_t qf[D / 16][4];
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    qf[kk][0] = qa_ptr ? ld_u32(qa_ptr + kk * 16 + 2 * tq) : 0u;
    qf[kk][1] = qb_ptr ? ld_u32(qb_ptr + kk * 16 + 2 * tq) : 0u;
    qf[kk][2] = qa_ptr ? ld_u32(qa_ptr + kk * 16 + 8 + 2 * tq) : 0u;
    qf[kk][3] = qb_ptr ? ld_u32(qb_ptr + kk * 16 + 8 + 2 * tq) : 0u;
  }

  float o[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;

  // the key blocks this CTA visits: cache chunks part, part+n_splits, ...; or the tree segment
  const __nv_bfloat16* kbase;
  const __nv_bfloat16* vbase;
  size_t key_stride;
  if (is_tree) {
    kbase = k_new + (static_cast<size_t>(b) * T * Hkv + g) * D;
    vbase = v_new + (static_cast<size_t>(b) * T * Hkv + g) * D;
    key_stride = static_cast<size_t>(Hkv) * D;
  } else {
    kbase = k_cache + (static_cast<size_t>(b) * Hkv + g) * Lmax * D;
    vbase = v_cache + (static_cast<size_t>(b) * Hkv + g) * Lmax * D;
    key_stride = D;
  }
  // enumerate blocks as (start key, end key) pairs
  auto block_range = [&](int it, int& k0, int& k1) -> bool {
    if (is_tree) {
      k0 = it * KB;
      k1 = min(T, k0 + KB);
      return k0 < T;
    }
    const int per_chunk = p.chunk / KB;
    const int c = part + (it / per_chunk) * p.n_splits;
    k0 = c * p.chunk + (it % per_chunk) * KB;
    k1 = min(min(L, c * p.chunk + p.chunk), k0 + KB);
    return k0 < L;
  };

  auto issue = [&](int buf, int k0, int k1) {
    const uint32_t dk = sK + buf * KB * D * 2, dv = sV + buf * KB * D * 2;
    for (int e = threadIdx.x; e < KB * NCH; e += blockDim.x) {
      const int j = e / NCH, c = e % NCH;
      const bool valid = k0 + j < k1;
      const size_t off = static_cast<size_t>(valid ? k0 + j : k0) * key_stride + c * 8;
      cp_async16(tile_addr<D>(dk, j, c), kbase + off, valid);
      cp_async16(tile_addr<D>(dv, j, c), vbase + off, valid);
    }
    cp_async_commit();
  };

  int k0, k1;
  bool have = block_range(0, k0, k1);
  if (have) issue(0, k0, k1);
  for (int it = 0; have; ++it) {
    int n0, n1;
    const bool have_next = block_range(it + 1, n0, n1);
    if (have_next) issue((it + 1) & 1, n0, n1);
    if (have_next) cp_async_wait<1>(); else cp_async_wait<0>();
    __syncthreads();
    const uint32_t tK = sK + (it & 1) * KB * D * 2, tV = sV + (it & 1) * KB * D * 2;

    // visibility words of this block for the two rows (tree segment)
    uint32_t wa0 = 0xffffffffu, wa1 = 0xffffffffu, wb0 = 0xffffffffu, wb1 = 0xffffffffu;
    if (is_tree) {
      const int w0 = k0 / 32;
      wa0 = node_a >= 0 ? tr.mask[static_cast<size_t>(node_a) * tr.mask_words + w0] : 0u;
      wb0 = node_b >= 0 ? tr.mask[static_cast<size_t>(node_b) * tr.mask_words + w0] : 0u;
      wa1 = (node_a >= 0 && w0 + 1 < tr.mask_words) ? tr.mask[static_cast<size_t>(node_a) * tr.mask_words + w0 + 1] : 0u;
      wb1 = (node_b >= 0 && w0 + 1 < tr.mask_words) ? tr.mask[static_cast<size_t>(node_b) * tr.mask_words + w0 + 1] : 0u;
    }
    const bool warp_active = __any_sync(0xffffffffu, (wa0 | wa1 | wb0 | wb1) != 0u) && row0 < R;

    if (warp_active) {
      float s[KB / 8][4];
#pragma unroll
      for (int nt = 0; nt < KB / 8; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
      for (int np = 0; np < KB / 16; ++np) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const int mat = lane >> 3, rr = lane & 7;
          uint32_t b0, b1, b2, b3;
          ldsm_x4(tile_addr<D>(tK, np * 16 + (mat >> 1) * 8 + rr, kk * 2 + (mat & 1)), b0, b1, b2, b3);
          mma_bf16(s[2 * np], qf[kk], b0, b1);
          mma_bf16(s[2 * np + 1], qf[kk], b2, b3);
        }
      }
      // scale + mask, row max
      float mx_a = -INFINITY, mx_b = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < KB / 8; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int kl = nt * 8 + 2 * tq + e;  // key offset in block
          const bool in = k0 + kl < k1;
          bool va = in, vb = in;
          if (is_tree) {
            va = in && (((kl < 32 ? wa0 >> kl : wa1 >> (kl - 32)) & 1u) != 0u);
            vb = in && (((kl < 32 ? wb0 >> kl : wb1 >> (kl - 32)) & 1u) != 0u);
          }
          s[nt][e] = va ? s[nt][e] * scale_log2 : -INFINITY;
          s[nt][2 + e] = vb ? s[nt][2 + e] * scale_log2 : -INFINITY;
          mx_a = fmaxf(mx_a, s[nt][e]);
          mx_b = fmaxf(mx_b, s[nt][2 + e]);
        }
      }
      mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 1));
      mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 2));
      mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 1));
      mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 2));
      const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
      const float al_a = mn_a == -INFINITY ? 1.f : exp2f(m_a - mn_a);
      const float al_b = mn_b == -INFINITY ? 1.f : exp2f(m_b - mn_b);
      m_a = mn_a;
      m_b = mn_b;
      float ps_a = 0.f, ps_b = 0.f;
#pragma unroll
      for (int nt = 0; nt < KB / 8; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          s[nt][e] = mn_a == -INFINITY ? 0.f : exp2f(s[nt][e] - mn_a);
          s[nt][2 + e] = mn_b == -INFINITY ? 0.f : exp2f(s[nt][2 + e] - mn_b);
          ps_a += s[nt][e];
          ps_b += s[nt][2 + e];
        }
      }
      l_a = l_a * al_a + ps_a;
      l_b = l_b * al_b + ps_b;
#pragma unroll
      for (int dn = 0; dn < D / 8; ++dn) {
        o[dn][0] *= al_a;
        o[dn][1] *= al_a;
        o[dn][2] *= al_b;
        o[dn][3] *= al_b;
      }
      // O += P V
#pragma unroll
      for (int kk = 0; kk < KB / 16; ++kk) {
        uint32_t pa[4];
        pa[0] = pack_bf16(s[2 * kk][0], s[2 * kk][1]);
        pa[1] = pack_bf16(s[2 * kk][2], s[2 * kk][3]);
        pa[2] = pack_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1]);
        pa[3] = pack_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
        for (int dp = 0; dp < D / 16; ++dp) {
          const int mat = lane >> 3, rr = lane & 7;
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(tile_addr<D>(tV, kk * 16 + (mat & 1) * 8 + rr, dp * 2 + (mat >> 1)), b0, b1, b2, b3);
          mma_bf16(o[2 * dp], pa, b0, b1);
          mma_bf16(o[2 * dp + 1], pa, b2, b3);
        }
      }
    }
    __syncthreads();
    k0 = n0;
    k1 = n1;
    have = have_next;
  }

  // partial results of this split
  l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
  l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
  l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
  l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);
  const size_t prow = (static_cast<size_t>(zb) * p.n_parts + part) * p.R_pad;
  if (ra < R) {
    float* dst = o_part + (prow + ra) * D;
#pragma unroll
    for (int dn = 0; dn < D / 8; ++dn)
      *reinterpret_cast<float2*>(dst + dn * 8 + 2 * tq) = make_float2(o[dn][0], o[dn][1]);
    if (tq == 0) ml_part[prow + ra] = make_float2(m_a, l_a);
  }
  if (rb < R) {
    float* dst = o_part + (prow + rb) * D;
#pragma unroll
    for (int dn = 0; dn < D / 8; ++dn)
      *reinterpret_cast<float2*>(dst + dn * 8 + 2 * tq) = make_float2(o[dn][2], o[dn][3]);
    if (tq == 0) ml_part[prow + rb] = make_float2(m_b, l_b);
  }
}

// Merge the splits: one warp per (request, node, query head).
template <int D>
__global__ void __launch_bounds__(256) attn_combine_kernel(int B, int T, int Hq, int Hkv, AttnPlan p,
                                                           const float* __restrict__ o_part,
                                                           const float2* __restrict__ ml_part, float* __restrict__ out,
                                                           int32_t* __restrict__ dev_status) {
  const int wid = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (wid >= B * T * Hq) return;
  const int hq = wid % Hq, i = (wid / Hq) % T, b = wid / (Hq * T);
  const int g = hq / p.G, row = i * p.G + hq % p.G;
  const size_t zrow = static_cast<size_t>(b * Hkv + g) * p.n_parts;
  float M = -INFINITY;
  for (int s = 0; s < p.n_parts; ++s) {
    const float2 ml = ml_part[(zrow + s) * p.R_pad + row];
    if (ml.y > 0.f) M = fmaxf(M, ml.x);
  }
  constexpr int PER = D / 32;
  float acc[PER] = {};
  float den = 0.f;
  for (int s = 0; s < p.n_parts; ++s) {
    const float2 ml = ml_part[(zrow + s) * p.R_pad + row];
    if (!(ml.y > 0.f)) continue;
    const float w = exp2f(ml.x - M);
    den += w * ml.y;
    const float* src = o_part + ((zrow + s) * p.R_pad + row) * D;
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] += w * src[lane + 32 * e];
  }
  float* dst = out + ((static_cast<size_t>(b) * T + i) * Hq + hq) * D;
  const float inv = 1.f / den;
#pragma unroll
  for (int e = 0; e < PER; ++e) dst[lane + 32 * e] = acc[e] * inv;
  if (lane == 0 && !(den > 0.f) && dev_status) atomicOr(dev_status + b, MEDUSA_DEV_NAN);
}

// Exact fp32 path: one CTA per (request, node, query head); scores in smem.
__global__ void __launch_bounds__(128) tree_attn_f32_kernel(medusa_tree_dev tr, const float* __restrict__ q,
                                                            const float* __restrict__ k_new,
                                                            const float* __restrict__ v_new,
                                                            const float* __restrict__ k_cache,
                                                            const float* __restrict__ v_cache,
                                                            const int32_t* __restrict__ kv_len, int Hq, int Hkv,
                                                            int D, int Lmax, float scale, float* __restrict__ out) {
  extern __shared__ float sc[];  // [Lmax + T]
  __shared__ float red[32];
  const int hq = blockIdx.x % Hq, i = (blockIdx.x / Hq) % tr.T, b = blockIdx.x / (Hq * tr.T);
  const int T = tr.T;
  const int g = hq / (Hq / Hkv);
  const int L = min(max(kv_len[b], 0), Lmax);
  const float* qv = q + ((static_cast<size_t>(b) * T + i) * Hq + hq) * D;
  const int n = L + T;
  for (int j = threadIdx.x; j < n; j += blockDim.x) {
    const float* kv;
    bool vis = true;
    if (j < L) {
      kv = k_cache + ((static_cast<size_t>(b) * Hkv + g) * Lmax + j) * D;
    } else {
      const int node = j - L;
      vis = (tr.mask[static_cast<size_t>(i) * tr.mask_words + node / 32] >> (node % 32)) & 1u;
      kv = k_new + ((static_cast<size_t>(b) * T + node) * Hkv + g) * D;
    }
    float s = 0.f;
    if (vis)
      for (int d = 0; d < D; ++d) s = fmaf(qv[d], kv[d], s);
    sc[j] = vis ? s * scale : -INFINITY;
  }
  __syncthreads();
  float mx = -INFINITY;
  for (int j = threadIdx.x; j < n; j += blockDim.x) mx = fmaxf(mx, sc[j]);
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
  __syncthreads();
  mx = -INFINITY;
  for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) mx = fmaxf(mx, red[w]);
  __syncthreads();
  float sum = 0.f;
  for (int j = threadIdx.x; j < n; j += blockDim.x) {
    const float e = expf(sc[j] - mx);
    sc[j] = e;
    sum += e;
  }
  sum = warp_sum(sum);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = sum;
  __syncthreads();
  sum = 0.f;
  for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) sum += red[w];
  const float inv = 1.f / sum;
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    float acc = 0.f;
    for (int j = 0; j < n; ++j) {
      if (sc[j] == 0.f) continue;
      const float* vv = j < L ? v_cache + ((static_cast<size_t>(b) * Hkv + g) * Lmax + j) * D
                              : v_new + ((static_cast<size_t>(b) * T + (j - L)) * Hkv + g) * D;
      acc = fmaf(sc[j], vv[d], acc);
    }
    out[((static_cast<size_t>(b) * T + i) * Hq + hq) * D + d] = acc * inv;
  }
}

}  // namespace

MEDUSA_API size_t medusa_tree_attention_workspace_size(const medusa_tree* tree, int32_t B, int32_t Hq, int32_t Hkv,
                                                       int32_t D, int32_t Lmax, int32_t kv_len_hint,
                                                       medusa_dtype dtype) {
  if (!tree || B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv || Lmax < 0) return 0;
  if (dtype == MEDUSA_F32) return 256;
  AttnPlan p = plan_attn(tree->T, B, Hq, Hkv, Lmax, kv_len_hint);
  return attn_ws_bytes(p, B, Hkv, D);
}

MEDUSA_API int medusa_tree_attention(const medusa_tree* tree, const void* q, const void* k_new, const void* v_new,
                                     const void* k_cache, const void* v_cache, const int32_t* kv_len, int32_t B,
                                     int32_t Hq, int32_t Hkv, int32_t D, int32_t Lmax, int32_t kv_len_hint,
                                     float scale, medusa_dtype dtype, float* out, void* ws, size_t ws_bytes,
                                     int32_t* dev_status, medusa_stream_t stream) {
  if (!tree || !q || !k_new || !v_new || !k_cache || !v_cache || !kv_len || !out) return MEDUSA_ERR_INVALID_ARG;
  if (B < 1 || B > MEDUSA_MAX_BATCH || Hq < 1 || Hkv < 1 || Lmax < 0 || Hq > 128) return MEDUSA_ERR_INVALID_ARG;
  if (dtype != MEDUSA_F32 && dtype != MEDUSA_BF16) return MEDUSA_ERR_INVALID_ARG;
  if (Hq % Hkv != 0 || (D != 64 && D != 128)) return MEDUSA_ERR_UNSUPPORTED;
  const void* ptrs[] = {q, k_new, v_new, k_cache, v_cache, kv_len, out};
  for (const void* x : ptrs)
    if (!aligned16(x)) return MEDUSA_ERR_ALIGNMENT;
  if ((ws && !aligned16(ws)) || (dev_status && !aligned16(dev_status))) return MEDUSA_ERR_ALIGNMENT;
  auto st = reinterpret_cast<cudaStream_t>(stream);
  const int T = tree->T;
  if (dtype == MEDUSA_F32) {
    const size_t smem = static_cast<size_t>(Lmax + T) * 4;
    if (smem > 200 * 1024) return MEDUSA_ERR_UNSUPPORTED;
    if (cudaFuncSetAttribute(tree_attn_f32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return MEDUSA_ERR_CUDA;
    tree_attn_f32_kernel<<<B * T * Hq, 128, smem, st>>>(
        tree->dev, static_cast<const float*>(q), static_cast<const float*>(k_new), static_cast<const float*>(v_new),
        static_cast<const float*>(k_cache), static_cast<const float*>(v_cache), kv_len, Hq, Hkv, D, Lmax, scale, out);
    MEDUSA_LAUNCH_CHECK();
    return MEDUSA_OK;
  }
  AttnPlan p = plan_attn(T, B, Hq, Hkv, Lmax, kv_len_hint);
  const size_t need = attn_ws_bytes(p, B, Hkv, D);
  if (!ws || ws_bytes < need) return MEDUSA_ERR_WORKSPACE;
  const size_t nrow = static_cast<size_t>(B) * Hkv * p.n_parts * p.R_pad;
  float* o_part = static_cast<float*>(ws);
  float2* ml_part = reinterpret_cast<float2*>(static_cast<char*>(ws) + align_up(nrow * D * 4, 256));
  const size_t smem = 4 * static_cast<size_t>(KB) * D * 2;
  dim3 grid(p.n_parts, p.n_qt, B * Hkv);
  const float scale_log2 = scale * 1.4426950408889634f;
  const int cthreads = 256;
  const int cblocks = cdiv(B * T * Hq, cthreads / 32);
  if (D == 128) {
    if (cudaFuncSetAttribute(tree_attn_bf16_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return MEDUSA_ERR_CUDA;
    tree_attn_bf16_kernel<128><<<grid, p.nwarps * 32, smem, st>>>(
        tree->dev, static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k_new),
        static_cast<const __nv_bfloat16*>(v_new), static_cast<const __nv_bfloat16*>(k_cache),
        static_cast<const __nv_bfloat16*>(v_cache), kv_len, Hq, Hkv, Lmax, p, scale_log2, o_part, ml_part);
    MEDUSA_LAUNCH_CHECK();
    attn_combine_kernel<128><<<cblocks, cthreads, 0, st>>>(B, T, Hq, Hkv, p, o_part, ml_part, out, dev_status);
  } else {
    if (cudaFuncSetAttribute(tree_attn_bf16_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return MEDUSA_ERR_CUDA;
    tree_attn_bf16_kernel<64><<<grid, p.nwarps * 32, smem, st>>>(
        tree->dev, static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k_new),
        static_cast<const __nv_bfloat16*>(v_new), static_cast<const __nv_bfloat16*>(k_cache),
        static_cast<const __nv_bfloat16*>(v_cache), kv_len, Hq, Hkv, Lmax, p, scale_log2, o_part, ml_part);
    MEDUSA_LAUNCH_CHECK();
    attn_combine_kernel<64><<<cblocks, cthreads, 0, st>>>(B, T, Hq, Hkv, p, o_part, ml_part, out, dev_status);
  }
  MEDUSA_LAUNCH_CHECK();
  return MEDUSA_OK;
}
