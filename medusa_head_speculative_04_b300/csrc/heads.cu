// Medusa heads (K1 + K2): u_k = h + SiLU(W1_k h + b1_k), z_k = W2_k u_k, per-head top-k.
//
// Ultralytics glossary "Medusa Heads", section "How the heads predict the next
// tokens": each head is one fully connected layer with SiLU and a residual
// connection followed by a bias-free projection onto the vocabulary, and every
// head reads the same last hidden state.  wiblog.cn "Medusa multi-head
// speculative decoding", section "Medusa decoding heads": each head outputs
// its top-k candidates.
//
// Both launches are HBM streams of weight rows (the batch has few rows, so
// the dot products run on CUDA cores from a shared-memory copy of the
// activations).  K2 fuses the top-k: every CTA keeps the top-k of its slice of
// the vocabulary, and the last CTA of a head (ticket counter) merges them.
// From kTcMinRows batch rows both products run on the tcgen05 GEMM of the
// verification pass instead; its epilogue keeps the top-k of every vocabulary
// tile and a small kernel merges the tiles' candidates per (row, head).
#include <algorithm>
#include <mutex>

#include "gemv.cuh"
#include "tc.cuh"
#include "tree.cuh"

using namespace medusa;

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRows = 4;  // most weight rows per warp pass
constexpr size_t kMaxXBytes = 96 * 1024;  // activation rows staged per launch

// Rows per warp pass (R) and 16-byte chunks per lane and row in flight (U):
// R*U = 16 loads in flight per lane.  With one or two activation rows a pass
// is one whole weight row (H = 4096 bf16 is 512 chunks = 16 per lane), so the
// warps' shares differ by at most one row; with more activation rows several
// weight rows share each staged activation chunk.
template <int BMAX> struct Pass {
  static constexpr int R = BMAX <= 2 ? 1 : BMAX <= 4 ? 2 : 4;
  static constexpr int U = BMAX <= 2 ? 16 : BMAX <= 4 ? 4 : 2;
};

// Work split.  Both launches size their grid to the CTAs that are resident at
// once (one wave).  K1 splits the weight rows evenly: first across CTAs, then
// across the warps of a CTA.  K2 gives every head (block) the same number of
// CTAs, so each CTA's rows lie inside one head and its top-k candidates belong
// to that head; with one or two activation rows and long heads it hands out a
// block's rows dynamically (a counter every warp takes its next rows from),
// else it splits them evenly like K1.
struct HeadsPlan {
  bool tc;      // vocabulary projection on the tensor cores (bf16, >= kTcMinRows rows, root given)
  bool fused;   // tc, with the top-k in the GEMM epilogue (k <= 16, candidates fit the merge CTA)
  int ntile;    // fused: vocabulary tiles per head, each contributing k candidates
  int nblk;     // K heads (+1 for the lm_head root block)
  int cph;      // CTAs per block (head)
  int rpc;      // most rows one K2 CTA holds
  int bgroup;   // batch rows per launch
  int fc_ctas;
};

constexpr size_t kSmemTwoPerSm = 110 * 1024;   // two CTAs per SM fit below this
constexpr size_t kSmemMax = 220 * 1024;        // per-CTA dynamic shared memory used at most

// K2 shared memory: staged activations, then one region holding first the
// CTA's logits [bmax][rpc] and, in the CTA that merges a head, every CTA's
// candidates [cph][topk] (values and ids), then per-warp and final top-k.
__host__ __device__ inline size_t vocab_region_floats(int bmax, int rpc, int cph, int topk) {
  const size_t z = static_cast<size_t>(bmax) * rpc, m = 2 * static_cast<size_t>(cph) * topk;
  return z > m ? z : m;
}
size_t vocab_smem_bytes(int nb, int bmax, int H, int esize, int rpc, int cph, int topk) {
  return align_up(static_cast<size_t>(nb) * H * esize, 16) +
         (vocab_region_floats(bmax, rpc, cph, topk) + 2 * kWarps * static_cast<size_t>(topk) +
          2 * static_cast<size_t>(topk)) * 4;
}

int bmax_of(int nb) { return nb == 1 ? 1 : nb == 2 ? 2 : nb <= 4 ? 4 : nb <= 8 ? 8 : 16; }

// From this many batch rows the CUDA-core dot products (B FMAs per weight
// element) fall behind the weight stream, and z_k = W2_k u_k runs as a tcgen05
// GEMM (M = batch rows, N = vocabulary) that writes the logits; K2 then only
// selects the top-k from them.
constexpr int kTcMinRows = 3;

// The merge of the tile candidates: [ntile*k] values and ids staged in shared
// memory, then the block-wide selection's per-warp and final lists.
size_t merge_smem_bytes(int ntile, int topk) {
  return (2 * static_cast<size_t>(ntile) * topk + 2 * static_cast<size_t>(kWarps) * topk + 2 * topk) * 4;
}
constexpr int kEpiTopkMaxK = 16;  // the GEMM epilogue keeps at most this many per tile

// Returns false when no split fits in shared memory.
bool plan_heads(int B, int H, int V, int K, int with_root, int esize, int topk, bool allow_tc, HeadsPlan* out) {
  HeadsPlan p{};
  const int sms = device_sm_count();
  p.tc = allow_tc && esize == 2 && !with_root && B >= kTcMinRows;
  p.nblk = K + (with_root ? 1 : 0);
  p.bgroup = static_cast<int>(std::min<size_t>(16, std::max<size_t>(1, kMaxXBytes / (static_cast<size_t>(H) * esize))));
  p.bgroup = std::min(p.bgroup, B);
  const int bm = bmax_of(p.bgroup);
  auto smem_of = [&](int cph) { return vocab_smem_bytes(p.bgroup, bm, H, esize, cdiv(V, cph), cph, topk); };
  // K2: one wave at two CTAs per SM (the GEMV is register-bound there), else one
  // wave at one CTA per SM, else as many CTAs as the per-CTA logit buffer needs
  int cph = std::max(1, std::min(2 * sms / p.nblk, V));
  if (smem_of(cph) > kSmemTwoPerSm) {
    cph = std::max(1, std::min(sms / p.nblk, V));
    const long fixed = static_cast<long>(align_up(static_cast<size_t>(p.bgroup) * H * esize, 16)) +
                       (2L * kWarps * topk + 2L * topk) * 4;
    const long budget = static_cast<long>(kSmemMax) - fixed;  // bytes for the logit/candidate region
    if (budget < 4L * bm) return false;
    const long rows_fit = budget / (4L * bm);
    cph = std::max<long>(cph, (V + rows_fit - 1) / rows_fit);
    cph = std::min(cph, V);
    if (smem_of(cph) > kSmemMax) return false;
  }
  p.cph = cph;
  p.rpc = cdiv(V, p.cph);
  const long fc_rows = static_cast<long>(K) * H;
  const size_t fc_smem = static_cast<size_t>(p.bgroup) * H * esize;
  const int fc_occ = fc_smem > kSmemTwoPerSm ? 1 : 2;
  p.fc_ctas = static_cast<int>(std::max(1L, std::min(static_cast<long>(sms) * fc_occ, fc_rows)));
  if (p.tc && topk <= kEpiTopkMaxK) {
    p.ntile = group_topk_tiles(B, K, V);
    p.fused = merge_smem_bytes(p.ntile, topk) <= kSmemMax;
  }
  *out = p;
  return true;
}

// Self-resetting counters in the workspace: per block a merge ticket and the
// row counter of K2's dynamic row split.
inline size_t counter_ints(const HeadsPlan& p) { return 2 * static_cast<size_t>(p.nblk); }

struct HeadsWs {
  void* u;
  float* z;    // [B, K, V] logits of the unfused tensor-core path when the caller keeps none
  float* zfc;  // [B, K*H] W1_k h of the tensor-core path
  float* cand_v;
  int* cand_i;
  int* counters;
  float* tile_v;  // fused: [B, K, ntile, topk] candidates of every vocabulary tile
  int* tile_i;
  size_t bytes;
};

HeadsWs carve_heads_ws(void* base, const HeadsPlan& p, int B, int H, int V, int K, int topk, int esize) {
  HeadsWs w{};
  size_t o = 0;
  auto take = [&](size_t n) { size_t s = o; o = align_up(o + n, 256); return s; };
  size_t ou = take(static_cast<size_t>(B) * K * H * esize);
  size_t ncand = p.fused ? 0 : static_cast<size_t>(p.nblk) * B * p.cph * topk;
  size_t ov = take(ncand * 4), oi = take(ncand * 4), oc = take(counter_ints(p) * 4);
  size_t oz = p.tc && !p.fused ? take(static_cast<size_t>(B) * K * V * 4) : 0;
  size_t ozf = p.tc ? take(static_cast<size_t>(B) * K * H * 4) : 0;
  const size_t ntc = p.fused ? static_cast<size_t>(B) * K * p.ntile * topk : 0;
  size_t otv = take(ntc * 4), oti = take(ntc * 4);
  char* c = static_cast<char*>(base);
  w.u = c ? c + ou : nullptr;
  w.z = c && p.tc && !p.fused ? reinterpret_cast<float*>(c + oz) : nullptr;
  w.zfc = c && p.tc ? reinterpret_cast<float*>(c + ozf) : nullptr;
  w.cand_v = c ? reinterpret_cast<float*>(c + ov) : nullptr;
  w.cand_i = c ? reinterpret_cast<int*>(c + oi) : nullptr;
  w.counters = c ? reinterpret_cast<int*>(c + oc) : nullptr;
  w.tile_v = c && p.fused ? reinterpret_cast<float*>(c + otv) : nullptr;
  w.tile_i = c && p.fused ? reinterpret_cast<int*>(c + oti) : nullptr;
  w.bytes = o;
  return w;
}

// Ask L2 for the first 4 KB of up to kRows weight rows (one 128-byte line per
// lane and row).  Weights are constant inputs of the step, so this may run
// before the wait on the preceding kernel.
template <typename T>
__device__ inline void prefetch_rows(const T* W, long row0, long rows, int H) {
  const int lane = threadIdx.x & 31;
  const long row_bytes = static_cast<long>(H) * sizeof(T);
  if (lane * 128L >= row_bytes) return;
  for (long r = row0; r < row0 + kRows && r < row0 + rows; ++r)
    asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char*>(W + r * H) + lane * 128));
}

// K2 takes the dynamic split when every warp gets at least this many rows.
constexpr int kDynMinRowsPerWarp = 16;

// Rows a warp takes from a dynamic row split at a time (a multiple of R).
template <int BMAX> struct Grab {
  static constexpr int G = 4 * Pass<BMAX>::R;
};

// Next G rows of a dynamic split: lane 0 adds to the counter, the warp gets the
// old value.  Issued one chunk ahead, so the atomic's round trip overlaps the
// rows being processed.
__device__ inline long grab_rows(int* ctr, int G) {
  long r = 0;
  if ((threadIdx.x & 31) == 0) r = atomicAdd(ctr, G);
  return r;
}

// Ask L2 for whole weight rows [row0, row0 + n) (n <= 32, one bulk prefetch per lane).
template <typename T>
__device__ inline void prefetch_whole_rows(const T* W, long row0, int n, long nrows, int H) {
  const int lane = threadIdx.x & 31;
  if (lane < n && row0 + lane < nrows)
    tc::prefetch_l2_bulk(W + (row0 + lane) * static_cast<long>(H), static_cast<uint32_t>(H * sizeof(T)));
}

// K1: rows [c*N/C, (c+1)*N/C) of W1 (flattened [K*H] rows) for CTA c, split
// evenly over its warps; each warp dots Pass::R rows at a time with nb rows of h.
template <typename T, int BMAX>
__global__ void __launch_bounds__(kThreads) heads_fc_kernel(const T* __restrict__ h, const T* __restrict__ W1,
                                                            const T* __restrict__ b1, int H, int K, int nb,
                                                            T* __restrict__ u) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  T* xs = reinterpret_cast<T*>(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long nrows = static_cast<long>(K) * H;
  const long c0 = blockIdx.x * nrows / gridDim.x, c1 = (blockIdx.x + 1) * nrows / gridDim.x;
  const long w0 = c0 + warp * (c1 - c0) / kWarps, w1 = c0 + (warp + 1) * (c1 - c0) / kWarps;
  prefetch_rows(W1, w0, w1 - w0, H);
  pdl_wait();
  pdl_trigger();
  stage_rows(xs, h, H, nb, H);
  __syncthreads();
  constexpr int R = Pass<BMAX>::R;
  for (long row0 = w0; row0 < w1; row0 += R) {
    const int valid = w1 - row0 < R ? static_cast<int>(w1 - row0) : R;
    // the biases of this pass load while the weight row streams in
    float bias[R];
#pragma unroll
    for (int r = 0; r < R; ++r) bias[r] = r < valid ? Elem<T>::to_f(b1[row0 + r]) : 0.f;
    float acc[R][BMAX];
    gemv_rows<T, BMAX, R, Pass<BMAX>::U>(W1, row0, valid, H, xs, nb, acc);
#pragma unroll
    for (int r = 0; r < R; ++r) {
#pragma unroll
      for (int b = 0; b < BMAX; ++b) {
        if (r < valid && b < nb && lane == ((r * BMAX + b) & 31)) {
          const long row = row0 + r;
          const int i = static_cast<int>(row % H);
          const float a = acc[r][b] + bias[r];
          const float silu = a / (1.0f + expf(-a));  // SiLU(a) = a * sigmoid(a)
          const float val = Elem<T>::to_f(xs[static_cast<size_t>(b) * H + i]) + silu;
          u[static_cast<size_t>(b) * nrows + row] = Elem<T>::from_f(val);
        }
      }
    }
  }
}

// K1 on the tensor-core path: u = h + SiLU(zfc + b1) for zfc = W1_k h from the
// GEMM, elementwise over [B, K*H] (the same arithmetic as heads_fc_kernel's
// epilogue).
template <typename T>
__global__ void __launch_bounds__(kThreads) heads_fc_act_kernel(const T* __restrict__ h, const T* __restrict__ b1,
                                                                const float* __restrict__ zfc, int B, int K, int H,
                                                                T* __restrict__ u) {
  pdl_wait();
  pdl_trigger();
  const long kh = static_cast<long>(K) * H, n = static_cast<long>(B) * kh;
  for (long e = blockIdx.x * static_cast<long>(blockDim.x) + threadIdx.x; e < n;
       e += static_cast<long>(gridDim.x) * blockDim.x) {
    const long b = e / kh, row = e % kh;
    const float a = zfc[e] + Elem<T>::to_f(b1[row]);
    const float silu = a / (1.0f + expf(-a));  // SiLU(a) = a * sigmoid(a)
    u[e] = Elem<T>::from_f(Elem<T>::to_f(h[b * H + row % H]) + silu);
  }
}

// K2: CTA j of block blk holds rows [j*V/cph, (j+1)*V/cph) of that block.
// Block blk < K is head blk (weights W2_blk, activations u[:, blk]); block K is
// lm_head on h (root).  FROMZ: the logits were computed by the tensor-core GEMM
// (zsrc [rows, K, V]) and the CTA only selects from its slice of them, copying
// it to head_logits when that is given.
template <typename T, int BMAX, bool FROMZ>
__global__ void __launch_bounds__(kThreads) heads_vocab_kernel(
    const T* __restrict__ h, const T* __restrict__ u, const T* __restrict__ W2, const T* __restrict__ lm_head,
    int B, int b0, int nb, int H, int V, int K, int topk, int rpc, int cph,
    float* __restrict__ head_logits, int32_t* __restrict__ topk_ids, float* __restrict__ topk_vals,
    int32_t* __restrict__ root_tok, float* __restrict__ cand_v, int* __restrict__ cand_i, int* __restrict__ counters,
    const float* __restrict__ zsrc) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int blk = blockIdx.x / cph, cta = blockIdx.x % cph;
  const bool is_root = blk == K;
  const int kk = is_root ? 1 : topk;
  const T* W = is_root ? lm_head : W2 + static_cast<size_t>(blk) * V * H;
  const T* x = is_root ? h + static_cast<size_t>(b0) * H : u + (static_cast<size_t>(b0) * K + blk) * H;
  const size_t x_stride = is_root ? H : static_cast<size_t>(K) * H;

  T* xs = reinterpret_cast<T*>(smem_raw);
  float* zs = reinterpret_cast<float*>(smem_raw + align_up(static_cast<size_t>(nb) * H * sizeof(T), 16));
  // the merge buffers reuse the logit region once the local top-k is out
  float* mv = zs;                                             // [cph * topk]
  int* mi = reinterpret_cast<int*>(mv + static_cast<size_t>(cph) * topk);
  float* sv = zs + vocab_region_floats(BMAX, rpc, cph, topk);  // [kWarps * topk]
  int* si = reinterpret_cast<int*>(sv + kWarps * topk);
  float* fv = reinterpret_cast<float*>(si + kWarps * topk);  // [topk] final
  int* fi = reinterpret_cast<int*>(fv + topk);
  __shared__ int s_last;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int v0 = static_cast<int>(static_cast<long>(cta) * V / cph);
  const int n = static_cast<int>(static_cast<long>(cta + 1) * V / cph) - v0;
  const int lr0 = warp * n / kWarps, lr1 = (warp + 1) * n / kWarps;  // this warp's local rows
  if (!FROMZ) prefetch_rows(W, v0 + lr0, lr1 - lr0, H);
  pdl_wait();
  pdl_trigger();
  if (FROMZ) {
    for (int e = threadIdx.x; e < nb * n; e += blockDim.x) {
      const int b = e / n, lr = e % n;
      const float z = zsrc[((static_cast<size_t>(b0) + b) * K + blk) * V + v0 + lr];
      zs[static_cast<size_t>(b) * rpc + lr] = z;
      if (head_logits) head_logits[(static_cast<size_t>(b0 + b) * K + blk) * V + v0 + lr] = z;
    }
  } else {
    stage_rows(xs, x, x_stride, nb, H);
  }
  __syncthreads();

  constexpr int R = Pass<BMAX>::R;
  for (int lr = lr0; lr < lr1 && !FROMZ; lr += R) {
    const int valid = min(R, lr1 - lr);
    float acc[R][BMAX];
    gemv_rows<T, BMAX, R, Pass<BMAX>::U>(W, static_cast<size_t>(v0 + lr), valid, H, xs, nb, acc);
#pragma unroll
    for (int r = 0; r < R; ++r) {
#pragma unroll
      for (int b = 0; b < BMAX; ++b) {
        if (r < valid && b < nb && lane == ((r * BMAX + b) & 31)) {
          zs[static_cast<size_t>(b) * rpc + lr + r] = acc[r][b];
          if (head_logits && !is_root)
            head_logits[(static_cast<size_t>(b0 + b) * K + blk) * V + v0 + lr + r] = acc[r][b];
        }
      }
    }
  }
  __syncthreads();

  // local top-k of this slice: one warp per batch row, rows side by side (a
  // block-wide selection per row would serialise the rows behind its barriers)
  for (int b = warp; b < nb; b += kWarps) {
    const size_t cb = ((static_cast<size_t>(blk) * B + b0 + b) * cph + cta) * topk;
    warp_topk_slice(zs + static_cast<size_t>(b) * rpc, nullptr, v0, n, kk, cand_v + cb, cand_i + cb,
                    __int_as_float(0x7fc00000));
  }

  // the last CTA of this block merges every slice's candidates
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(counters + blk, 1) == cph - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int b = 0; b < nb; ++b) {
    const size_t base = (static_cast<size_t>(blk) * B + b0 + b) * cph * topk;
    const int m = cph * kk;
    for (int e = threadIdx.x; e < m; e += blockDim.x) {
      const int c = e / kk, t = e % kk;
      mv[e] = __ldcg(cand_v + base + static_cast<size_t>(c) * topk + t);
      mi[e] = __ldcg(cand_i + base + static_cast<size_t>(c) * topk + t);
    }
    __syncthreads();
    block_topk(mv, mi, 0, m, kk, fv, fi, sv, si);
    if (is_root) {
      if (threadIdx.x == 0) root_tok[b0 + b] = fi[0];
    } else {
      for (int t = threadIdx.x; t < topk; t += blockDim.x) {
        topk_ids[(static_cast<size_t>(b0 + b) * K + blk) * topk + t] = fi[t];
        topk_vals[(static_cast<size_t>(b0 + b) * K + blk) * topk + t] = fv[t];
      }
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) counters[blk] = 0;  // ready for the next launch
}

// K2 for one or two activation rows: the rows of block blk (head blk's W2, or
// lm_head for the root) in a dynamic split over the block's CTAs (every warp
// takes the next G rows from the block's counter until none are left), so the
// launch ends with little tail.  Each warp keeps the top-k of the rows it took,
// per activation row, as a list spread over lanes 0..k-1 (value descending, equal
// values by the lower id, NaN never taken): a row's logit enters if it beats the
// k-th entry.  The CTA then merges its warps' lists into k candidates, and the
// last CTA of the block (ticket) merges the CTAs' candidates, as in the static
// split, and resets the block's counters.
template <int BMAX>
size_t vocab_dyn_smem_bytes(int nb, int H, int esize, int cph, int topk) {
  return align_up(static_cast<size_t>(nb) * H * esize, 16) +
         (2 * static_cast<size_t>(cph) * topk + 2 * kWarps * static_cast<size_t>(topk) + 2 * static_cast<size_t>(topk) +
          2 * static_cast<size_t>(BMAX) * kWarps * topk) * 4;
}

template <typename T, int BMAX>
__global__ void __launch_bounds__(kThreads, 2) heads_vocab_dyn_kernel(
    const T* __restrict__ h, const T* __restrict__ u, const T* __restrict__ W2, const T* __restrict__ lm_head,
    int B, int b0, int nb, int H, int V, int K, int topk, int cph, float* __restrict__ head_logits,
    int32_t* __restrict__ topk_ids, float* __restrict__ topk_vals, int32_t* __restrict__ root_tok,
    float* __restrict__ cand_v, int* __restrict__ cand_i, int* __restrict__ counters) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int nblk = gridDim.x / cph;
  const int blk = blockIdx.x / cph, cta = blockIdx.x % cph;
  const bool is_root = blk == K;
  const int kk = is_root ? 1 : topk;
  const T* W = is_root ? lm_head : W2 + static_cast<size_t>(blk) * V * H;
  const T* x = is_root ? h + static_cast<size_t>(b0) * H : u + (static_cast<size_t>(b0) * K + blk) * H;
  const size_t x_stride = is_root ? H : static_cast<size_t>(K) * H;
  int* rowctr = counters + nblk + blk;

  T* xs = reinterpret_cast<T*>(smem_raw);
  float* mv = reinterpret_cast<float*>(smem_raw + align_up(static_cast<size_t>(nb) * H * sizeof(T), 16));
  int* mi = reinterpret_cast<int*>(mv + static_cast<size_t>(cph) * topk);  // [cph * topk] merge
  float* sv = reinterpret_cast<float*>(mi + static_cast<size_t>(cph) * topk);  // [kWarps * topk]
  int* si = reinterpret_cast<int*>(sv + kWarps * topk);
  float* fv = reinterpret_cast<float*>(si + kWarps * topk);  // [topk] final
  int* fi = reinterpret_cast<int*>(fv + topk);
  float* wv = reinterpret_cast<float*>(fi + topk);  // [BMAX][kWarps * topk] the warps' lists, kk apart
  int* wi = reinterpret_cast<int*>(wv + BMAX * kWarps * topk);
  __shared__ int s_last;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int R = Pass<BMAX>::R, G = Grab<BMAX>::G;
  // the block's counter was reset by this kernel's previous launch, which
  // completed before any kernel ahead of this one did
  long r0 = __shfl_sync(0xffffffffu, grab_rows(rowctr, G), 0);
  prefetch_whole_rows(W, r0, G, V, H);
  pdl_wait();
  pdl_trigger();
  stage_rows(xs, x, x_stride, nb, H);
  __syncthreads();

  float lv[BMAX], tv[BMAX];
  int li[BMAX], ti[BMAX];
#pragma unroll
  for (int b = 0; b < BMAX; ++b) {
    lv[b] = tv[b] = -INFINITY;
    li[b] = ti[b] = 0x7fffffff;
  }
  while (r0 < V) {
    const long nx = grab_rows(rowctr, G);
    const int r1 = static_cast<int>(r0 + G < V ? r0 + G : V);
    for (int row0 = static_cast<int>(r0); row0 < r1; row0 += R) {
      const int valid = min(R, r1 - row0);
      float acc[R][BMAX];
      gemv_rows<T, BMAX, R, Pass<BMAX>::U>(W, static_cast<size_t>(row0), valid, H, xs, nb, acc);
#pragma unroll
      for (int r = 0; r < R; ++r) {
#pragma unroll
        for (int b = 0; b < BMAX; ++b) {
          if (r < valid && b < nb) {
            const float z = acc[r][b];  // every lane holds the row's logit
            const int id = row0 + r;
            if (head_logits && !is_root && lane == 0)
              head_logits[(static_cast<size_t>(b0 + b) * K + blk) * V + id] = z;
            if (better(z, id, tv[b], ti[b])) {
              // fewer than kk entries are ahead of it: shift the rest down one lane
              const int pos = __popc(__ballot_sync(0xffffffffu, lane < kk && better(lv[b], li[b], z, id)));
              const float uv = __shfl_up_sync(0xffffffffu, lv[b], 1);
              const int ui = __shfl_up_sync(0xffffffffu, li[b], 1);
              if (lane == pos) {
                lv[b] = z;
                li[b] = id;
              } else if (lane > pos && lane < kk) {
                lv[b] = uv;
                li[b] = ui;
              }
              tv[b] = __shfl_sync(0xffffffffu, lv[b], kk - 1);
              ti[b] = __shfl_sync(0xffffffffu, li[b], kk - 1);
            }
          }
        }
      }
    }
    r0 = __shfl_sync(0xffffffffu, nx, 0);
  }

  // the warps' lists side by side (unfilled entries NaN, never taken), then one
  // warp per activation row merges them into the CTA's candidates
#pragma unroll
  for (int b = 0; b < BMAX; ++b) {
    if (b < nb && lane < kk) {
      const bool filled = li[b] != 0x7fffffff;
      wv[b * kWarps * topk + warp * kk + lane] = filled ? lv[b] : __int_as_float(0x7fc00000);
      wi[b * kWarps * topk + warp * kk + lane] = filled ? li[b] : -1;
    }
  }
  __syncthreads();
  for (int b = warp; b < nb; b += kWarps) {
    float* v = wv + b * kWarps * topk;
    int* ids = wi + b * kWarps * topk;
    const size_t cb = ((static_cast<size_t>(blk) * B + b0 + b) * cph + cta) * topk;
    warp_topk_slice(v, ids, 0, kWarps * kk, kk, cand_v + cb, cand_i + cb, __int_as_float(0x7fc00000));
  }

  // the last CTA of this block merges every CTA's candidates
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(counters + blk, 1) == cph - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int b = 0; b < nb; ++b) {
    const size_t base = (static_cast<size_t>(blk) * B + b0 + b) * cph * topk;
    const int m = cph * kk;
    for (int e = threadIdx.x; e < m; e += blockDim.x) {
      const int c = e / kk, t = e % kk;
      mv[e] = __ldcg(cand_v + base + static_cast<size_t>(c) * topk + t);
      mi[e] = __ldcg(cand_i + base + static_cast<size_t>(c) * topk + t);
    }
    __syncthreads();
    block_topk(mv, mi, 0, m, kk, fv, fi, sv, si);
    if (is_root) {
      if (threadIdx.x == 0) root_tok[b0 + b] = fi[0];
    } else {
      for (int t = threadIdx.x; t < topk; t += blockDim.x) {
        topk_ids[(static_cast<size_t>(b0 + b) * K + blk) * topk + t] = fi[t];
        topk_vals[(static_cast<size_t>(b0 + b) * K + blk) * topk + t] = fv[t];
      }
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {  // ready for the next launch
    counters[blk] = 0;
    *rowctr = 0;
  }
}

template <typename T, int BMAX>
int launch_fc(const HeadsPlan& p, const HeadsWs& w, const T* h, const T* W1, const T* b1, int b0, int nb, int H,
              int K, cudaStream_t st) {
  const size_t xbytes = align_up(static_cast<size_t>(nb) * H * sizeof(T), 16);
  auto fc = heads_fc_kernel<T, BMAX>;
  if (!ensure_dyn_smem(fc, xbytes))
    return MEDUSA_ERR_CUDA;
  if (launch_pdl(fc, dim3(p.fc_ctas), dim3(kThreads), xbytes, st, h + static_cast<size_t>(b0) * H, W1, b1, H, K, nb,
                 static_cast<T*>(w.u) + static_cast<size_t>(b0) * K * H) != cudaSuccess) {
    (void)cudaGetLastError();
    return MEDUSA_ERR_CUDA;
  }
  MEDUSA_LAUNCH_CHECK();
  return MEDUSA_OK;
}

template <typename T, int BMAX, bool FROMZ>
int launch_vocab(const HeadsPlan& p, const HeadsWs& w, const T* h, const T* W2, const T* lm, int B, int b0, int nb,
                 int H, int V, int K, int topk, float* head_logits, int32_t* topk_ids, float* topk_vals,
                 int32_t* root_tok, const float* zsrc, cudaStream_t st) {
  if constexpr (!FROMZ && BMAX <= 2) {
    // short heads keep the static split: the counter's round trips would cost more than the tail
    if (static_cast<long>(V) >= static_cast<long>(kDynMinRowsPerWarp) * p.cph * kWarps) {
      const size_t smem = vocab_dyn_smem_bytes<BMAX>(nb, H, sizeof(T), p.cph, topk);
      auto vk = heads_vocab_dyn_kernel<T, BMAX>;
      if (!ensure_dyn_smem(vk, smem))
        return MEDUSA_ERR_CUDA;
      if (launch_pdl(vk, dim3(p.nblk * p.cph), dim3(kThreads), smem, st, h, static_cast<const T*>(w.u), W2, lm, B,
                     b0, nb, H, V, K, topk, p.cph, head_logits, topk_ids, topk_vals, root_tok, w.cand_v, w.cand_i,
                     w.counters) != cudaSuccess) {
        (void)cudaGetLastError();
        return MEDUSA_ERR_CUDA;
      }
      MEDUSA_LAUNCH_CHECK();
      return MEDUSA_OK;
    }
  }
  const size_t smem = vocab_smem_bytes(nb, BMAX, H, sizeof(T), p.rpc, p.cph, topk);
  auto vk = heads_vocab_kernel<T, BMAX, FROMZ>;
  if (!ensure_dyn_smem(vk, smem))
    return MEDUSA_ERR_CUDA;
  if (launch_pdl(vk, dim3(p.nblk * p.cph), dim3(kThreads), smem, st, h, static_cast<const T*>(w.u), W2, lm, B, b0, nb,
                 H, V, K, topk, p.rpc, p.cph, head_logits, topk_ids, topk_vals, root_tok, w.cand_v, w.cand_i,
                 w.counters, zsrc) != cudaSuccess) {
    (void)cudaGetLastError();
    return MEDUSA_ERR_CUDA;
  }
  MEDUSA_LAUNCH_CHECK();
  return MEDUSA_OK;
}

template <typename T, bool FROMZ>
int launch_vocab_nb(const HeadsPlan& p, const HeadsWs& w, const T* h, const T* W2, const T* lm, int B, int b0,
                    int nb, int H, int V, int K, int topk, float* hl, int32_t* ids, float* vals, int32_t* root,
                    const float* zsrc, cudaStream_t st) {
  if (nb == 1) return launch_vocab<T, 1, FROMZ>(p, w, h, W2, lm, B, b0, nb, H, V, K, topk, hl, ids, vals, root, zsrc, st);
  if (nb == 2) return launch_vocab<T, 2, FROMZ>(p, w, h, W2, lm, B, b0, nb, H, V, K, topk, hl, ids, vals, root, zsrc, st);
  if (nb <= 4) return launch_vocab<T, 4, FROMZ>(p, w, h, W2, lm, B, b0, nb, H, V, K, topk, hl, ids, vals, root, zsrc, st);
  if (nb <= 8) return launch_vocab<T, 8, FROMZ>(p, w, h, W2, lm, B, b0, nb, H, V, K, topk, hl, ids, vals, root, zsrc, st);
  return launch_vocab<T, 16, FROMZ>(p, w, h, W2, lm, B, b0, nb, H, V, K, topk, hl, ids, vals, root, zsrc, st);
}

template <typename T>
int launch_fc_nb(const HeadsPlan& p, const HeadsWs& w, const T* h, const T* W1, const T* b1, int b0, int nb, int H,
                 int K, cudaStream_t st) {
  if (nb == 1) return launch_fc<T, 1>(p, w, h, W1, b1, b0, nb, H, K, st);
  if (nb == 2) return launch_fc<T, 2>(p, w, h, W1, b1, b0, nb, H, K, st);
  if (nb <= 4) return launch_fc<T, 4>(p, w, h, W1, b1, b0, nb, H, K, st);
  if (nb <= 8) return launch_fc<T, 8>(p, w, h, W1, b1, b0, nb, H, K, st);
  return launch_fc<T, 16>(p, w, h, W1, b1, b0, nb, H, K, st);
}

// Merge of the fused path: CTA (b, head) takes the top-k of the ntile*topk
// candidates its vocabulary tiles left (unfilled ones are NaN and never taken).
__global__ void __launch_bounds__(kThreads) topk_merge_kernel(const float* __restrict__ tile_v,
                                                              const int* __restrict__ tile_i, int K, int ntile,
                                                              int topk, int32_t* __restrict__ topk_ids,
                                                              float* __restrict__ topk_vals) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int n = ntile * topk;
  float* mv = reinterpret_cast<float*>(smem_raw);
  int* mi = reinterpret_cast<int*>(mv + n);
  float* sv = reinterpret_cast<float*>(mi + n);  // [kWarps * topk]
  int* si = reinterpret_cast<int*>(sv + kWarps * topk);
  float* fv = reinterpret_cast<float*>(si + kWarps * topk);
  int* fi = reinterpret_cast<int*>(fv + topk);
  pdl_wait();
  pdl_trigger();
  const size_t base = static_cast<size_t>(blockIdx.x) * n;  // blockIdx.x = b * K + head
  for (int e = threadIdx.x; e < n; e += blockDim.x) {
    mv[e] = tile_v[base + e];
    mi[e] = tile_i[base + e];
  }
  __syncthreads();
  block_topk(mv, mi, 0, n, topk, fv, fi, sv, si);
  for (int t = threadIdx.x; t < topk; t += blockDim.x) {
    topk_ids[static_cast<size_t>(blockIdx.x) * topk + t] = fi[t];
    topk_vals[static_cast<size_t>(blockIdx.x) * topk + t] = fv[t];
  }
}

int launch_topk_merge(const HeadsPlan& p, const HeadsWs& w, int rows, int K, int topk, int32_t* ids, float* vals,
                      cudaStream_t st) {
  const size_t smem = merge_smem_bytes(p.ntile, topk);
  if (!ensure_dyn_smem(topk_merge_kernel, smem))
    return MEDUSA_ERR_CUDA;
  if (launch_pdl(topk_merge_kernel, dim3(rows * K), dim3(kThreads), smem, st, static_cast<const float*>(w.tile_v),
                 static_cast<const int*>(w.tile_i), K, p.ntile, topk, ids, vals) != cudaSuccess) {
    (void)cudaGetLastError();
    return MEDUSA_ERR_CUDA;
  }
  MEDUSA_LAUNCH_CHECK();
  return MEDUSA_OK;
}

// The tensor-core path (bf16 only): u = h + SiLU(W1_k h + b1_k) with W1 as one
// [K*H, H] GEMM plus an elementwise launch, then z_k = W2_k u_k as K grouped
// GEMMs: fused, with the tiles' top-k candidates into the workspace (and the
// logits into z when z is given); else the logits into z.
int tc_heads(const HeadsPlan&, const HeadsWs&, const float*, const float*, const float*, const float*, int, int, int,
             int, int, float*, cudaStream_t) {
  return MEDUSA_ERR_UNSUPPORTED;
}
int tc_heads(const HeadsPlan& p, const HeadsWs& w, const __nv_bfloat16* h, const __nv_bfloat16* W1,
             const __nv_bfloat16* b1, const __nv_bfloat16* W2, int B, int H, int V, int K, int topk, float* z,
             cudaStream_t st) {
  int rc = launch_group_logits_bf16(h, B, 1, W1, H, K * H, w.zfc, st);
  if (rc != MEDUSA_OK) return rc;
  const long n = static_cast<long>(B) * K * H;
  const int blocks = static_cast<int>(std::min<long>(cdiv(static_cast<int>(std::min<long>(n, 1L << 30)), kThreads),
                                                     4L * device_sm_count()));
  if (launch_pdl(heads_fc_act_kernel<__nv_bfloat16>, dim3(blocks), dim3(kThreads), 0, st, h, b1,
                 static_cast<const float*>(w.zfc), B, K, H, static_cast<__nv_bfloat16*>(w.u)) != cudaSuccess) {
    (void)cudaGetLastError();
    return MEDUSA_ERR_CUDA;
  }
  MEDUSA_LAUNCH_CHECK();
  if (p.fused)
    return launch_group_topk_bf16(w.u, B, K, W2, H, V, topk, w.tile_v, w.tile_i, z, st);
  return launch_group_logits_bf16(w.u, B, K, W2, H, V, z, st);
}

template <typename T>
int heads_dispatch(const HeadsPlan& p, const HeadsWs& w, const T* h, const T* W1, const T* b1, const T* W2,
                   const T* lm, int B, int H, int V, int K, int topk, float* hl, int32_t* ids, float* vals,
                   int32_t* root, cudaStream_t st) {
  if (p.tc) {
    // u and z = W2_k u_k on the tensor cores, then the top-k of z
    if (p.fused) {
      const int rc = tc_heads(p, w, h, W1, b1, W2, B, H, V, K, topk, hl, st);
      return rc != MEDUSA_OK ? rc : launch_topk_merge(p, w, B, K, topk, ids, vals, st);
    }
    float* z = hl ? hl : w.z;
    int rc = tc_heads(p, w, h, W1, b1, W2, B, H, V, K, topk, z, st);
    if (rc != MEDUSA_OK) return rc;
    for (int b0 = 0; b0 < B; b0 += p.bgroup) {
      rc = launch_vocab_nb<T, true>(p, w, h, W2, lm, B, b0, std::min(p.bgroup, B - b0), H, V, K, topk, nullptr, ids,
                                    vals, root, z, st);
      if (rc != MEDUSA_OK) return rc;
    }
    return MEDUSA_OK;
  }
  for (int b0 = 0; b0 < B; b0 += p.bgroup) {
    const int nb = std::min(p.bgroup, B - b0);
    int rc = launch_fc_nb(p, w, h, W1, b1, b0, nb, H, K, st);
    if (rc == MEDUSA_OK)
      rc = launch_vocab_nb<T, false>(p, w, h, W2, lm, B, b0, nb, H, V, K, topk, hl, ids, vals, root, nullptr, st);
    if (rc != MEDUSA_OK) return rc;
  }
  return MEDUSA_OK;
}

}  // namespace

MEDUSA_API size_t medusa_heads_topk_workspace_size(int32_t B, int32_t H, int32_t V, int32_t K, int32_t topk,
                                                   int32_t with_lm_head, medusa_dtype dtype) {
  if (B < 1 || H < 8 || V < 1 || K < 1 || topk < 1) return 0;
  const int es = dtype == MEDUSA_BF16 ? 2 : 4;
  HeadsPlan p;
  if (!plan_heads(B, H, V, K, with_lm_head, es, topk, true, &p)) return 0;
  return carve_heads_ws(nullptr, p, B, H, V, K, topk, es).bytes;
}

MEDUSA_API int medusa_heads_topk(const void* h, const void* w1, const void* b1, const void* w2, const void* lm_head,
                                 int32_t B, int32_t H, int32_t V, int32_t K, int32_t topk, medusa_dtype dtype,
                                 float* head_logits, int32_t* topk_ids, float* topk_vals, int32_t* root_tok,
                                 void* ws, size_t ws_bytes, medusa_stream_t stream) {
  if (!h || !w1 || !b1 || !w2 || !topk_ids || !topk_vals || !root_tok) return MEDUSA_ERR_INVALID_ARG;
  if (dtype != MEDUSA_F32 && dtype != MEDUSA_BF16) return MEDUSA_ERR_INVALID_ARG;
  if (B < 1 || B > MEDUSA_MAX_BATCH || K < 1 || V < 1 || H < 8 || topk < 1 || topk > MEDUSA_MAX_TOPK || topk > V)
    return MEDUSA_ERR_INVALID_ARG;
  if (H % 8 != 0) return MEDUSA_ERR_UNSUPPORTED;
  const void* ptrs[] = {h, w1, b1, w2, topk_ids, topk_vals, root_tok, ws};
  for (const void* q : ptrs)
    if (q && !aligned16(q)) return MEDUSA_ERR_ALIGNMENT;
  if ((lm_head && !aligned16(lm_head)) || (head_logits && !aligned16(head_logits))) return MEDUSA_ERR_ALIGNMENT;
  const int es = dtype == MEDUSA_BF16 ? 2 : 4;
  HeadsPlan p;
  if (!plan_heads(B, H, V, K, lm_head != nullptr, es, topk, true, &p)) return MEDUSA_ERR_UNSUPPORTED;
  HeadsWs w = carve_heads_ws(ws, p, B, H, V, K, topk, es);
  if (!ws || ws_bytes < w.bytes) return MEDUSA_ERR_WORKSPACE;
  auto st = reinterpret_cast<cudaStream_t>(stream);
  if (dtype == MEDUSA_BF16)
    return heads_dispatch(p, w, static_cast<const __nv_bfloat16*>(h), static_cast<const __nv_bfloat16*>(w1),
                          static_cast<const __nv_bfloat16*>(b1), static_cast<const __nv_bfloat16*>(w2),
                          static_cast<const __nv_bfloat16*>(lm_head), B, H, V, K, topk, head_logits, topk_ids,
                          topk_vals, root_tok, st);
  return heads_dispatch(p, w, static_cast<const float*>(h), static_cast<const float*>(w1),
                        static_cast<const float*>(b1), static_cast<const float*>(w2),
                        static_cast<const float*>(lm_head), B, H, V, K, topk, head_logits, topk_ids, topk_vals,
                        root_tok, st);
}

// ---------------------------------------------------------------------------
// medusa_heads_topk_tree: the next step's candidates from the verification
// pass's hidden states.  wiblog.cn "Medusa multi-head speculative decoding",
// section "Inference flow in an online chat service": the pass that scores the
// candidates also yields what the next round's candidates come from, with no
// extra forward pass; Ultralytics glossary "Medusa Heads", section "Tree
// attention and accepting tokens": the accepted branch continues the sequence.
// Only the accepted node's heads are kept, and acceptance is known when this
// runs, so each request's accepted row x[b, best_node[b]] is gathered first and
// the heads run on those B rows (the same outputs as running them on every
// node and keeping the accepted one, for B rows of work instead of B*T).
// ---------------------------------------------------------------------------
namespace {

// xg[b] = x[b, clamp(best[b])] (16-byte chunks).
template <typename T>
__global__ void __launch_bounds__(256) gather_rows_kernel(const T* __restrict__ x, const int32_t* __restrict__ best,
                                                          int Tn, int H, T* __restrict__ xg) {
  const int b = blockIdx.x;
  pdl_wait();
  pdl_trigger();
  const int node = min(max(best[b], 0), Tn - 1);
  constexpr int E = Elem<T>::kPer16B;
  const uint4* src = reinterpret_cast<const uint4*>(x + (static_cast<size_t>(b) * Tn + node) * H);
  uint4* dst = reinterpret_cast<uint4*>(xg + static_cast<size_t>(b) * H);
  for (int c = threadIdx.x; c < H / E; c += blockDim.x) dst[c] = src[c];
}

struct TreeHeadsWs {
  void* xg;      // [B, H] the accepted rows
  HeadsWs hw;    // the heads on those rows
  size_t bytes;
};

TreeHeadsWs carve_tree_heads_ws(void* base, const HeadsPlan& p, int B, int H, int V, int K, int topk, int es) {
  TreeHeadsWs w{};
  const size_t gx = align_up(static_cast<size_t>(B) * H * es, 256);
  char* c = static_cast<char*>(base);
  w.xg = c;
  w.hw = carve_heads_ws(c ? c + gx : nullptr, p, B, H, V, K, topk, es);
  w.bytes = gx + w.hw.bytes;
  return w;
}

template <typename T>
int tree_heads_dispatch(const HeadsPlan& p, const TreeHeadsWs& w, const T* x, const T* W1, const T* b1, const T* W2,
                        const int32_t* best, int B, int Tn, int H, int V, int K, int topk, float* hl, int32_t* ids,
                        float* vals, cudaStream_t st) {
  if (launch_pdl(gather_rows_kernel<T>, dim3(B), dim3(256), 0, st, x, best, Tn, H, static_cast<T*>(w.xg)) !=
      cudaSuccess) {
    (void)cudaGetLastError();
    return MEDUSA_ERR_CUDA;
  }
  MEDUSA_LAUNCH_CHECK();
  return heads_dispatch(p, w.hw, static_cast<const T*>(w.xg), W1, b1, W2, static_cast<const T*>(nullptr), B, H, V,
                        K, topk, hl, ids, vals, static_cast<int32_t*>(nullptr), st);
}

}  // namespace

MEDUSA_API size_t medusa_heads_topk_tree_workspace_size(const medusa_tree* tree, int32_t B, int32_t H, int32_t V,
                                                        int32_t K, int32_t topk, medusa_dtype dtype) {
  if (!tree || B < 1 || H < 8 || V < 1 || K < 1 || topk < 1) return 0;
  const int es = dtype == MEDUSA_BF16 ? 2 : 4;
  HeadsPlan p;
  if (!plan_heads(B, H, V, K, 0, es, topk, true, &p)) return 0;
  return carve_tree_heads_ws(nullptr, p, B, H, V, K, topk, es).bytes;
}

MEDUSA_API int medusa_heads_topk_tree(const medusa_tree* tree, const void* x, const void* w1, const void* b1,
                                      const void* w2, const int32_t* best_node, int32_t B, int32_t H, int32_t V,
                                      int32_t K, int32_t topk, medusa_dtype dtype, float* head_logits,
                                      int32_t* topk_ids, float* topk_vals, void* ws, size_t ws_bytes,
                                      medusa_stream_t stream) {
  if (!tree || !x || !w1 || !b1 || !w2 || !best_node || !topk_ids || !topk_vals) return MEDUSA_ERR_INVALID_ARG;
  if (dtype != MEDUSA_F32 && dtype != MEDUSA_BF16) return MEDUSA_ERR_INVALID_ARG;
  if (B < 1 || B > MEDUSA_MAX_BATCH || K < 1 || V < 1 || H < 8 || topk < 1 || topk > MEDUSA_MAX_TOPK || topk > V)
    return MEDUSA_ERR_INVALID_ARG;
  if (H % 8 != 0) return MEDUSA_ERR_UNSUPPORTED;
  const void* ptrs[] = {x, w1, b1, w2, best_node, topk_ids, topk_vals};
  for (const void* q : ptrs)
    if (!aligned16(q)) return MEDUSA_ERR_ALIGNMENT;
  if ((head_logits && !aligned16(head_logits)) || (ws && !aligned16(ws))) return MEDUSA_ERR_ALIGNMENT;
  const int es = dtype == MEDUSA_BF16 ? 2 : 4;
  const int Tn = tree->T;
  HeadsPlan p;
  if (!plan_heads(B, H, V, K, 0, es, topk, true, &p)) return MEDUSA_ERR_UNSUPPORTED;
  TreeHeadsWs w = carve_tree_heads_ws(ws, p, B, H, V, K, topk, es);
  if (!ws || ws_bytes < w.bytes) return MEDUSA_ERR_WORKSPACE;
  auto st = reinterpret_cast<cudaStream_t>(stream);
  if (dtype == MEDUSA_BF16)
    return tree_heads_dispatch(p, w, static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(w1),
                               static_cast<const __nv_bfloat16*>(b1), static_cast<const __nv_bfloat16*>(w2), best_node,
                               B, Tn, H, V, K, topk, head_logits, topk_ids, topk_vals, st);
  return tree_heads_dispatch(p, w, static_cast<const float*>(x), static_cast<const float*>(w1),
                             static_cast<const float*>(b1), static_cast<const float*>(w2), best_node, B, Tn, H, V, K,
                             topk, head_logits, topk_ids, topk_vals, st);
}

// ---------------------------------------------------------------------------
// medusa_heads_topk_noalloc: the same heads step for callers that must not
// allocate device memory.  Its scratch (u, per-CTA candidates, tickets) is a
// fixed array compiled into this library, so the caller passes only inputs
// and outputs.  The array lives on every GPU that loads the library until the
// process exits, and all calls share it: calls that overlap on the GPU race.
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kNoAllocScratchBytes = static_cast<size_t>(MEDUSA_NOALLOC_SCRATCH_BYTES);
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_heads_scratch[kNoAllocScratchBytes];

// Device address of g_heads_scratch on the current device.  Host code only has
// a host-side stand-in under that name, so the address is looked up with the
// device current.  A call made outside a stream capture looks it up afresh (a
// host-side table lookup in the CUDA runtime; the first one on a device also
// loads this library's device code), so a device reset or a recreated context
// never leaves a stale address behind; a call made while `st` is capturing
// reuses the address found by the last call on that device outside a capture.
int heads_scratch_address(cudaStream_t st, void** out) {
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    (void)cudaGetLastError();
    return MEDUSA_ERR_CUDA;
  }
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cap) != cudaSuccess) {
    (void)cudaGetLastError();
    return MEDUSA_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (cap == cudaStreamCaptureStatusNone) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_heads_scratch) != cudaSuccess || !p) {
      (void)cudaGetLastError();
      return MEDUSA_ERR_CUDA;
    }
    addr[dev] = p;
  }
  if (!addr[dev]) return MEDUSA_ERR_CUDA;  // first call on this device made inside a capture
  *out = addr[dev];
  return MEDUSA_OK;
}

}  // namespace

MEDUSA_API int medusa_heads_topk_noalloc(const void* h, const void* w1, const void* b1, const void* w2,
                                         const void* lm_head, int32_t B, int32_t H, int32_t V, int32_t K,
                                         int32_t topk, medusa_dtype dtype, float* head_logits, int32_t* topk_ids,
                                         float* topk_vals, int32_t* root_tok, medusa_stream_t stream) {
  if (!h || !w1 || !b1 || !w2 || !topk_ids || !topk_vals || !root_tok) return MEDUSA_ERR_INVALID_ARG;
  if (dtype != MEDUSA_F32 && dtype != MEDUSA_BF16) return MEDUSA_ERR_INVALID_ARG;
  if (B < 1 || B > MEDUSA_MAX_BATCH || K < 1 || V < 1 || H < 8 || topk < 1 || topk > MEDUSA_MAX_TOPK || topk > V)
    return MEDUSA_ERR_INVALID_ARG;
  if (H % 8 != 0) return MEDUSA_ERR_UNSUPPORTED;
  const void* ptrs[] = {h, w1, b1, w2, topk_ids, topk_vals, root_tok};
  for (const void* q : ptrs)
    if (!aligned16(q)) return MEDUSA_ERR_ALIGNMENT;
  if ((lm_head && !aligned16(lm_head)) || (head_logits && !aligned16(head_logits))) return MEDUSA_ERR_ALIGNMENT;
  const int es = dtype == MEDUSA_BF16 ? 2 : 4;
  HeadsPlan p;
  if (!plan_heads(B, H, V, K, lm_head != nullptr, es, topk, false, &p)) return MEDUSA_ERR_UNSUPPORTED;
  if (carve_heads_ws(nullptr, p, B, H, V, K, topk, es).bytes > kNoAllocScratchBytes) return MEDUSA_ERR_SCRATCH_LIMIT;
  auto st = reinterpret_cast<cudaStream_t>(stream);
  void* scratch = nullptr;
  const int rc = heads_scratch_address(st, &scratch);
  if (rc != MEDUSA_OK) return rc;
  HeadsWs w = carve_heads_ws(scratch, p, B, H, V, K, topk, es);
  // the ticket counters must start at zero whatever an earlier call left behind
  if (cudaMemsetAsync(w.counters, 0, counter_ints(p) * sizeof(int), st) != cudaSuccess) {
    (void)cudaGetLastError();
    return MEDUSA_ERR_CUDA;
  }
  if (dtype == MEDUSA_BF16)
    return heads_dispatch(p, w, static_cast<const __nv_bfloat16*>(h), static_cast<const __nv_bfloat16*>(w1),
                          static_cast<const __nv_bfloat16*>(b1), static_cast<const __nv_bfloat16*>(w2),
                          static_cast<const __nv_bfloat16*>(lm_head), B, H, V, K, topk, head_logits, topk_ids,
                          topk_vals, root_tok, st);
  return heads_dispatch(p, w, static_cast<const float*>(h), static_cast<const float*>(w1),
                        static_cast<const float*>(b1), static_cast<const float*>(w2),
                        static_cast<const float*>(lm_head), B, H, V, K, topk, head_logits, topk_ids, topk_vals,
                        root_tok, st);
}
