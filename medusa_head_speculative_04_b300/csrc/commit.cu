// KV commit (K7): the accepted path's K/V rows join the cache.
//
// Ultralytics glossary "Medusa Heads", section "Tree attention and accepting
// tokens": the longest branch the model accepts is kept; wiblog.cn "Medusa
// multi-head speculative decoding", section "Inference flow in an online chat
// service": the accepted tokens are emitted and the next round starts from the
// last of them.  The tree pass already computed the K/V rows of every node, so
// keeping a branch means copying the rows of its nodes (depth 0..a) to cache
// positions kv_len..kv_len+a.  One CTA per request: it reads kv_len once,
// finds the path from the winner's ancestor-mask row, copies with 16-byte
// vectors and only then publishes the new length.
#include "tree.cuh"

using namespace medusa;

namespace {

constexpr int kCommitThreads = 512;
constexpr int kCommitUnroll = 4;

__global__ void __launch_bounds__(kCommitThreads) kv_commit_kernel(
    medusa_tree_dev tr, const uint4* __restrict__ k_new, const uint4* __restrict__ v_new, uint4* __restrict__ k_cache,
    uint4* __restrict__ v_cache, int32_t* __restrict__ kv_len, const int32_t* __restrict__ best_node, int Hkv,
    int row_vecs, int Lmax, int32_t* __restrict__ dev_status) {
  __shared__ int chain[MEDUSA_MAX_DEPTH + 1];
  __shared__ int s_best, s_n, s_L;
  extern __shared__ int16_t s_dep[];  // [T] depths: constant, read before the wait
  const int b = blockIdx.x;
  const int T = tr.T, mw = tr.mask_words;
  for (int t = threadIdx.x; t < T; t += blockDim.x) s_dep[t] = static_cast<int16_t>(tr.depth[t]);
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x == 0) {
    int best = best_node[b];
    if (best < 0 || best >= T) best = 0;
    const int a = s_dep[best];
    const int L = kv_len[b];
    s_best = best;
    s_L = L;
    s_n = (L < 0 || L + a + 1 > Lmax) ? -1 : a + 1;
    if (s_n < 0 && dev_status) atomicOr(dev_status + b, MEDUSA_DEV_KV_OVERFLOW);
  }
  __syncthreads();
  // the kept path root..best, by depth, read off best's ancestor-mask row
  const int best = s_best;
  for (int t = threadIdx.x; t < T; t += blockDim.x)
    if ((tr.mask[static_cast<size_t>(best) * mw + t / 32] >> (t % 32)) & 1u) chain[s_dep[t]] = t;
  __syncthreads();
  const int n = s_n, L = s_L;
  if (n < 0) return;
  // element e -> (depth d, kv head g, 16-byte vector j of a row); all loads of a
  // round are issued before its stores
  const int per_d = Hkv * row_vecs;
  const int total = n * per_d;
  for (int e0 = threadIdx.x; e0 < total; e0 += blockDim.x * kCommitUnroll) {
    uint4 kr[kCommitUnroll], vr[kCommitUnroll];
#pragma unroll
    for (int u = 0; u < kCommitUnroll; ++u) {
      const int e = e0 + u * blockDim.x;
      if (e < total) {
        const int d = e / per_d, g = (e / row_vecs) % Hkv, j = e % row_vecs;
        const size_t src = ((static_cast<size_t>(b) * T + chain[d]) * Hkv + g) * row_vecs + j;
        kr[u] = k_new[src];
        vr[u] = v_new[src];
      }
    }
#pragma unroll
    for (int u = 0; u < kCommitUnroll; ++u) {
      const int e = e0 + u * blockDim.x;
      if (e < total) {
        const int d = e / per_d, g = (e / row_vecs) % Hkv, j = e % row_vecs;
        const size_t dst = ((static_cast<size_t>(b) * Hkv + g) * Lmax + L + d) * row_vecs + j;
        k_cache[dst] = kr[u];
        v_cache[dst] = vr[u];
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) kv_len[b] = L + n;
}

}  // namespace

MEDUSA_API int medusa_kv_commit(const medusa_tree* tree, const void* k_new, const void* v_new, void* k_cache,
                                void* v_cache, int32_t* kv_len, const int32_t* best_node, int32_t B, int32_t Hkv,
                                int32_t D, int32_t Lmax, medusa_dtype dtype, int32_t* dev_status,
                                medusa_stream_t stream) {
  if (!tree || !k_new || !v_new || !k_cache || !v_cache || !kv_len || !best_node) return MEDUSA_ERR_INVALID_ARG;
  if (B < 1 || B > MEDUSA_MAX_BATCH || Hkv < 1 || D < 1 || Lmax < 0) return MEDUSA_ERR_INVALID_ARG;
  if (dtype != MEDUSA_F32 && dtype != MEDUSA_BF16) return MEDUSA_ERR_INVALID_ARG;
  const int es = dtype == MEDUSA_BF16 ? 2 : 4;
  if ((D * es) % 16 != 0) return MEDUSA_ERR_UNSUPPORTED;
  const void* ptrs[] = {k_new, v_new, k_cache, v_cache, kv_len, best_node};
  for (const void* q : ptrs)
    if (!aligned16(q)) return MEDUSA_ERR_ALIGNMENT;
  if (dev_status && !aligned16(dev_status)) return MEDUSA_ERR_ALIGNMENT;
  if (launch_pdl(kv_commit_kernel, dim3(B), dim3(kCommitThreads), static_cast<size_t>(tree->T) * 2,
                 reinterpret_cast<cudaStream_t>(stream),
                 tree->dev, static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new),
                 static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), kv_len, best_node, Hkv, D * es / 16, Lmax,
                 dev_status) != cudaSuccess) {
    (void)cudaGetLastError();
    return MEDUSA_ERR_CUDA;
  }
  MEDUSA_LAUNCH_CHECK();
  return MEDUSA_OK;
}
