// Candidate tree: host-side table construction (once per tree) and the per-step
// expansion kernel (K3) that turns per-head top-k candidates into tree tokens.
//
// The tree is fixed and regular, so its ancestor mask is prepared once and
// cached (wiblog.cn "Medusa multi-head speculative decoding", section "Tree
// attention"); every depth-d node takes head d's candidates, the same ones
// under every branch (Ultralytics glossary "Medusa Heads", section "Tree
// attention and accepting tokens").
#include <algorithm>
#include <atomic>
#include <cstring>
#include <map>
#include <vector>

#include "tree.cuh"

using namespace medusa;

namespace medusa {
static std::atomic<uint64_t> g_launches{0};
void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

int device_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return 148;
  }
  return n;
}
}  // namespace medusa

MEDUSA_API uint64_t medusa_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

MEDUSA_API const char* medusa_status_string(int s) {
  switch (s) {
    case MEDUSA_OK: return "ok";
    case MEDUSA_ERR_INVALID_ARG: return "invalid argument";
    case MEDUSA_ERR_ALIGNMENT: return "device pointer not 16-byte aligned";
    case MEDUSA_ERR_UNSUPPORTED: return "unsupported shape";
    case MEDUSA_ERR_WORKSPACE: return "workspace missing or too small";
    case MEDUSA_ERR_CUDA: return "CUDA call or launch failed";
    case MEDUSA_ERR_SCRATCH_LIMIT: return "shape needs more scratch than the built-in array holds";
    default: return "unknown status";
  }
}

MEDUSA_API int medusa_tree_create(const int32_t* ranks_flat, const int32_t* lens, int32_t n_choices,
                                  medusa_tree** out) {
  if (!out || n_choices < 0 || (n_choices > 0 && (!ranks_flat || !lens))) return MEDUSA_ERR_INVALID_ARG;
  *out = nullptr;
  if (1 + n_choices > MEDUSA_MAX_NODES) return MEDUSA_ERR_INVALID_ARG;
  std::vector<std::vector<int32_t>> cs(n_choices);
  size_t off = 0;
  for (int i = 0; i < n_choices; ++i) {
    if (lens[i] < 1 || lens[i] > MEDUSA_MAX_DEPTH) return MEDUSA_ERR_INVALID_ARG;
    cs[i].assign(ranks_flat + off, ranks_flat + off + lens[i]);
    off += lens[i];
    for (int32_t r : cs[i])
      if (r < 0 || r >= MEDUSA_MAX_TOPK) return MEDUSA_ERR_INVALID_ARG;
  }
  // canonical order: by depth, then lexicographic rank tuple
  std::sort(cs.begin(), cs.end(), [](const std::vector<int32_t>& a, const std::vector<int32_t>& b) {
    if (a.size() != b.size()) return a.size() < b.size();
    return a < b;
  });
  for (int i = 1; i < n_choices; ++i)
    if (cs[i] == cs[i - 1]) return MEDUSA_ERR_INVALID_ARG;  // duplicate
  std::map<std::vector<int32_t>, int32_t> index;
  index[{}] = 0;
  for (int i = 0; i < n_choices; ++i) index[cs[i]] = i + 1;

  auto* t = new medusa_tree();
  const int T = n_choices + 1;
  t->T = T;
  t->parent.assign(T, -1);
  t->depth.assign(T, 0);
  t->rank.assign(T, -1);
  t->child_start.assign(T, 0);
  t->child_count.assign(T, 0);
  for (int i = 0; i < n_choices; ++i) {
    std::vector<int32_t> pre(cs[i].begin(), cs[i].end() - 1);
    auto it = index.find(pre);
    if (it == index.end()) { delete t; return MEDUSA_ERR_INVALID_ARG; }  // not prefix-closed
    const int node = i + 1;
    t->parent[node] = it->second;
    t->depth[node] = static_cast<int32_t>(cs[i].size());
    t->rank[node] = cs[i].back();
    t->dmax = std::max(t->dmax, t->depth[node]);
    int d = t->depth[node] - 1;
    t->max_rank[d] = std::max(t->max_rank[d], t->rank[node]);
  }
  // children are contiguous: same prefix, consecutive in lexicographic order
  for (int node = 1; node < T; ++node) {
    int p = t->parent[node];
    if (t->child_count[p] == 0) t->child_start[p] = node;
    t->child_count[p]++;
  }
  t->mask_words = cdiv(T, 32);
  t->mask.assign(static_cast<size_t>(T) * t->mask_words, 0u);
  for (int i = 0; i < T; ++i)
    for (int a = i; a >= 0; a = t->parent[a]) t->mask[static_cast<size_t>(i) * t->mask_words + a / 32] |= 1u << (a % 32);
  for (int i = 0; i < T; ++i)
    if (t->child_count[i] == 0) t->leaf.push_back(i);
  t->P = static_cast<int32_t>(t->leaf.size());
  const int W = t->dmax + 1;
  t->paths.assign(static_cast<size_t>(t->P) * W, -1);
  t->first_path.assign(T, -1);
  for (int p = 0; p < t->P; ++p) {
    for (int a = t->leaf[p]; a >= 0; a = t->parent[a]) {
      t->paths[static_cast<size_t>(p) * W + t->depth[a]] = a;
      if (t->first_path[a] < 0) t->first_path[a] = p;
    }
  }

  // one device block holding every table
  const size_t n_i32 = 6 * static_cast<size_t>(T) + t->paths.size() + t->leaf.size();
  const size_t bytes_i32 = align_up(n_i32 * 4, 256);
  const size_t bytes = bytes_i32 + t->mask.size() * 4;
  cudaGetDevice(&t->device);
  if (cudaMalloc(&t->dev_block, bytes) != cudaSuccess) { delete t; return MEDUSA_ERR_CUDA; }
  std::vector<int32_t> host(n_i32);
  size_t o = 0;
  auto put = [&](const std::vector<int32_t>& v) { size_t s = o; std::copy(v.begin(), v.end(), host.begin() + o); o += v.size(); return s; };
  size_t o_parent = put(t->parent), o_depth = put(t->depth), o_rank = put(t->rank);
  size_t o_cs = put(t->child_start), o_cc = put(t->child_count), o_paths = put(t->paths), o_leaf = put(t->leaf);
  size_t o_fp = put(t->first_path);
  auto* base = static_cast<int32_t*>(t->dev_block);
  auto* mask = reinterpret_cast<uint32_t*>(static_cast<char*>(t->dev_block) + bytes_i32);
  if (cudaMemcpy(base, host.data(), n_i32 * 4, cudaMemcpyHostToDevice) != cudaSuccess ||
      cudaMemcpy(mask, t->mask.data(), t->mask.size() * 4, cudaMemcpyHostToDevice) != cudaSuccess) {
    cudaFree(t->dev_block);
    delete t;
    return MEDUSA_ERR_CUDA;
  }
  t->dev = medusa_tree_dev{T, t->P, t->dmax, t->mask_words, base + o_parent, base + o_depth, base + o_rank,
                           base + o_cs, base + o_cc, mask, base + o_paths, base + o_leaf, base + o_fp};
  *out = t;
  return MEDUSA_OK;
}

const std::vector<uint64_t>& tree_tile_visibility(medusa_tree* t, int G, int rpt) {
  std::lock_guard<std::mutex> lock(t->vis_mu);
  auto key = std::make_pair(G, rpt);
  auto it = t->vis_cache.find(key);
  if (it != t->vis_cache.end()) return it->second;
  const int R = t->T * G, n_qt = cdiv(R, rpt), mw = t->mask_words;
  std::vector<uint64_t> v(n_qt, 0);
  for (int qt = 0; qt < n_qt; ++qt) {
    const int r0 = qt * rpt, r1 = std::min(R, r0 + rpt);
    for (int node = r0 / G; node <= (r1 - 1) / G; ++node)
      for (int w = 0; w < mw; ++w)
        if (t->mask[static_cast<size_t>(node) * mw + w]) v[qt] |= 1ull << (w >> 1);
  }
  return t->vis_cache.emplace(key, std::move(v)).first->second;
}

MEDUSA_API int medusa_tree_get_info(const medusa_tree* t, medusa_tree_info* info) {
  if (!t || !info) return MEDUSA_ERR_INVALID_ARG;
  std::memset(info, 0, sizeof(*info));
  info->T = t->T;
  info->P = t->P;
  info->dmax = t->dmax;
  info->mask_words = t->mask_words;
  for (int d = 0; d < MEDUSA_MAX_DEPTH; ++d) info->max_rank[d] = t->max_rank[d];
  return MEDUSA_OK;
}

MEDUSA_API int medusa_tree_query(const medusa_tree* t, int32_t* T, int32_t* P, int32_t* dmax, int32_t* topk_per_depth) {
  if (!t) return MEDUSA_ERR_INVALID_ARG;
  if (T) *T = t->T;
  if (P) *P = t->P;
  if (dmax) *dmax = t->dmax;
  if (topk_per_depth)
    for (int d = 0; d < MEDUSA_MAX_DEPTH; ++d) topk_per_depth[d] = d < t->dmax ? t->max_rank[d] + 1 : 0;
  return MEDUSA_OK;
}

MEDUSA_API int medusa_tree_copy_tables(const medusa_tree* t, int32_t* parent, int32_t* depth, int32_t* rank,
                                       uint32_t* mask, int32_t* paths) {
  if (!t) return MEDUSA_ERR_INVALID_ARG;
  if (parent) std::copy(t->parent.begin(), t->parent.end(), parent);
  if (depth) std::copy(t->depth.begin(), t->depth.end(), depth);
  if (rank) std::copy(t->rank.begin(), t->rank.end(), rank);
  if (mask) std::copy(t->mask.begin(), t->mask.end(), mask);
  if (paths) std::copy(t->paths.begin(), t->paths.end(), paths);
  return MEDUSA_OK;
}

MEDUSA_API void medusa_tree_destroy(medusa_tree* t) {
  if (!t) return;
  if (t->dev_block) {
    int cur = 0;
    cudaGetDevice(&cur);
    if (cur != t->device) cudaSetDevice(t->device);
    cudaFree(t->dev_block);
    if (cur != t->device) cudaSetDevice(cur);
  }
  delete t;
}

// --------------------------------------------------------------------------
// K3: tree expansion.  One CTA per request, one thread per node (strided).
// --------------------------------------------------------------------------
__global__ void build_tree_kernel(medusa_tree_dev tr, const int32_t* __restrict__ root_tok,
                                  const int32_t* __restrict__ topk_ids, int K, int topk,
                                  const int32_t* __restrict__ kv_len, int32_t* __restrict__ tokens,
                                  int32_t* __restrict__ pos, int32_t* __restrict__ candidates,
                                  int32_t* __restrict__ dev_status) {
  const int b = blockIdx.x;
  const int T = tr.T;
  // depth and rank of every node: constant tables, read before the wait
  extern __shared__ int16_t s_tab[];  // [2][T]
  int16_t* s_dep = s_tab;
  int16_t* s_rank = s_tab + T;
  for (int i = threadIdx.x; i < T; i += blockDim.x) {
    s_dep[i] = static_cast<int16_t>(tr.depth[i]);
    s_rank[i] = static_cast<int16_t>(tr.rank[i]);
  }
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  const int32_t L = kv_len[b];
  const int32_t root = root_tok[b];
  bool bad = root < 0;
  auto token_of = [&](int node) -> int32_t {
    const int d = s_dep[node];
    if (d == 0) return root;
    return topk_ids[(static_cast<size_t>(b) * K + (d - 1)) * topk + s_rank[node]];
  };
  for (int i = threadIdx.x; i < T; i += blockDim.x) {
    const int32_t tok = token_of(i);
    bad |= tok < 0;
    tokens[static_cast<size_t>(b) * T + i] = tok;
    pos[static_cast<size_t>(b) * T + i] = L + s_dep[i];
  }
  if (candidates) {
    const int W = tr.dmax + 1;
    for (int e = threadIdx.x; e < tr.P * W; e += blockDim.x) {
      const int node = tr.paths[e];
      candidates[static_cast<size_t>(b) * tr.P * W + e] = node >= 0 ? token_of(node) : -1;
    }
  }
  if (bad && dev_status) atomicOr(dev_status + b, MEDUSA_DEV_BAD_TOKEN);
}

MEDUSA_API int medusa_build_tree(const medusa_tree* tree, const int32_t* root_tok, const int32_t* topk_ids,
                                 int32_t B, int32_t K, int32_t topk, const int32_t* kv_len,
                                 int32_t* tree_tokens, int32_t* position_ids, int32_t* candidates,
                                 int32_t* dev_status, medusa_stream_t stream) {
  if (!tree || !root_tok || !topk_ids || !kv_len || !tree_tokens || !position_ids) return MEDUSA_ERR_INVALID_ARG;
  if (B < 1 || B > MEDUSA_MAX_BATCH || K < 1 || topk < 1 || topk > MEDUSA_MAX_TOPK) return MEDUSA_ERR_INVALID_ARG;
  if (tree->dmax > K) return MEDUSA_ERR_INVALID_ARG;
  for (int d = 0; d < tree->dmax; ++d)
    if (tree->max_rank[d] >= topk) return MEDUSA_ERR_INVALID_ARG;
  if (!aligned16(root_tok) || !aligned16(topk_ids) || !aligned16(kv_len) || !aligned16(tree_tokens) ||
      !aligned16(position_ids) || (candidates && !aligned16(candidates)) || (dev_status && !aligned16(dev_status)))
    return MEDUSA_ERR_ALIGNMENT;
  if (launch_pdl(build_tree_kernel, dim3(B), dim3(256), static_cast<size_t>(tree->T) * 4,
                 reinterpret_cast<cudaStream_t>(stream), tree->dev,
                 root_tok, topk_ids, K, topk, kv_len, tree_tokens, position_ids, candidates, dev_status) != cudaSuccess) {
    (void)cudaGetLastError();
    return MEDUSA_ERR_CUDA;
  }
  MEDUSA_LAUNCH_CHECK();
  return MEDUSA_OK;
}
