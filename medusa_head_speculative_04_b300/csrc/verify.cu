// Verification (K5) and typical acceptance (K6).
//
// wiblog.cn "Medusa multi-head speculative decoding", section "Inference flow
// in an online chat service": the original model computes, in one pass, the
// probability of every candidate token in the tree; section "Typical
// acceptance": a candidate is kept when its probability exceeds the minimum of
// a hard threshold and an entropy-dependent threshold, the first token is
// always taken greedily, the longest passing prefix is output, and at
// temperature zero the scheme is greedy decoding.  cnnetsun.cn "Medusa safety
// considerations", section "Posterior probability evaluation":
// evaluate_posterior(logits, candidates, temperature, posterior_threshold,
// posterior_alpha) -> best_candidate, accept_length.
//
// K5 (bf16): logits = X lm_head^T for every tree node is a GEMM with M = tree
// rows (B*T) and N = vocabulary.  tcgen05.mma accumulates a 128 x BN tile in
// TMEM from TMA-fed, 128-byte-swizzled shared-memory stages (one producer
// thread, one MMA thread).  The epilogue (4 warps, one TMEM lane = one tree
// node each) never writes the logits unless asked: it reduces its vocabulary
// tile to (max, argmax, sum of exp, sum of exp * logit) at the temperature and
// picks out the logits of the node's children tokens.
// K5 (fp32): CUDA-core GEMV into a logits buffer, then the same statistics.
// K6a merges the per-tile statistics of every node; K6b decides acceptance,
// the longest kept prefix, the next root, one CTA per request.
#include <algorithm>
#include <mutex>

#include "gemv.cuh"
#include "tc.cuh"
#include "tree.cuh"

using namespace medusa;

namespace medusa {

EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

bool make_tmap_bf16(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tmap_bf16_3d(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                       uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box1, uint32_t box2) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
  cuuint32_t box[3] = {64, box1, box2};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace medusa

namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int F32_TILE = 256;  // vocabulary columns per statistics tile on the fp32 path

struct VerifyPlan {
  int R, BN, n_mt, n_nt;
};

VerifyPlan plan_verify(int B, int T, int V, medusa_dtype dt) {
  VerifyPlan p{};
  p.R = B * T;
  if (dt == MEDUSA_BF16) {
    p.n_mt = cdiv(p.R, BM);
    if (p.n_mt == 1)
      p.BN = std::min(256, std::max(16, cdiv(cdiv(V, 148), 16) * 16));
    else
      p.BN = 256;
    p.n_nt = cdiv(V, p.BN);
  } else {
    p.n_mt = 1;
    p.BN = F32_TILE;
    p.n_nt = cdiv(V, F32_TILE);
  }
  return p;
}

struct VerifyWs {
  float4* part;      // [R, n_nt] (max, sum exp, sum exp*y, argmax bits)
  float* child_z;    // [R] logit of node c's token under its parent (indexed by c)
  float4* rowst;     // [R] merged statistics
  int* tickets;      // [B] CTAs done with a request's nodes (self-resetting)
  float* zbuf;       // fp32 path: [R, V] logits when the caller gives none
  size_t bytes;
};

VerifyWs carve_verify_ws(void* base, const VerifyPlan& p, int V, medusa_dtype dt) {
  VerifyWs w{};
  size_t o = 0;
  auto take = [&](size_t n) { size_t s = o; o = align_up(o + n, 256); return s; };
  size_t op = take(static_cast<size_t>(p.R) * p.n_nt * 16), oc = take(static_cast<size_t>(p.R) * 4),
         orow = take(static_cast<size_t>(p.R) * 16), otk = take(static_cast<size_t>(p.R) * 4);
  size_t oz = dt == MEDUSA_F32 ? take(static_cast<size_t>(p.R) * V * 4) : 0;
  char* c = static_cast<char*>(base);
  if (c) {
    w.part = reinterpret_cast<float4*>(c + op);
    w.child_z = reinterpret_cast<float*>(c + oc);
    w.rowst = reinterpret_cast<float4*>(c + orow);
    w.tickets = reinterpret_cast<int*>(c + otk);
    w.zbuf = dt == MEDUSA_F32 ? reinterpret_cast<float*>(c + oz) : nullptr;
  }
  w.bytes = o;
  return w;
}

struct EpiArgs {
  int R, V, T, n_nt;
  const int32_t* tokens;
  medusa_tree_dev tr;
  float inv_tau;  // 0 at temperature 0 (statistics beyond max/argmax skipped)
  float* logits;
  float4* part;
  float* child_z;
  int32_t* dev_status;
};

// ------------------------------------------------------------------------
// K5, bf16: tcgen05 GEMM with the statistics epilogue.
// Warps 0..kEpiWarps-1 run the epilogue (warp w reads TMEM lanes 32*(w%4)..
// and the (w/4)-th of kEpiWarps/4 column groups of the tile); the next warp
// streams lm_head tiles, the next issues the MMAs and owns TMEM, the last
// streams the tree rows X.
// lm_head (from HBM) and X (from L2, shared by every CTA) run in separate
// rings: a deep one for the weight stream, a shallow one for X, whose stage
// holds only the xr rows the tile has (xr <= 128; the MMA's reads of rows
// xr..127 land in the next stage's bytes and only feed accumulator rows that
// are never read).
// ------------------------------------------------------------------------
constexpr int kMaxStages = 8;
constexpr int kEpiWarps = 8;
constexpr int kWarpW = kEpiWarps, kWarpMma = kEpiWarps + 1, kWarpX = kEpiWarps + 2;
constexpr int kTcThreads = (kEpiWarps + 3) * 32;
constexpr int kColGroups = kEpiWarps / 4;
constexpr size_t kHalfXchgBytes = (kColGroups - 1) * BM * 5 * 4;  // per-row statistics of groups 1..


struct TcShape {
  int BN, xr, sw, sx;  // vocab tile, X rows per stage, lm_head stages, X stages
};

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Running statistics of one row over a 32-column chunk v[0..nv): maximum and
// its first column (tree reduction), then, at temperature > 0, the sums
// s = sum 2^y2 and w2 = sum 2^y2 * y2 with y2 = (z - m) * k2, k2 = log2(e) /
// temperature, rescaled when the maximum grows.  NaN never wins the maximum.
__device__ inline void chunk_stats(const float (&v)[32], int nv, int col0, float k2, bool tempered, float& m,
                                   int& arg, float& s, float& w2, bool& nan_seen) {
  float t[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const bool in = j < nv;
    nan_seen |= in && v[j] != v[j];
    t[j] = (in && v[j] == v[j]) ? v[j] : -INFINITY;
  }
  float tv[16];
  int ti[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const bool take = t[j + 16] > t[j];
    tv[j] = take ? t[j + 16] : t[j];
    ti[j] = take ? j + 16 : j;
  }
#pragma unroll
  for (int h = 8; h >= 1; h >>= 1) {
#pragma unroll
    for (int j = 0; j < h; ++j) {
      const bool take = tv[j + h] > tv[j];
      tv[j] = take ? tv[j + h] : tv[j];
      ti[j] = take ? ti[j + h] : ti[j];
    }
  }
  const float cm = tv[0];
  if (cm > m) {
    if (tempered && s > 0.f) {
      const float d2 = (m - cm) * k2;
      const float sc = exp2f(d2);
      w2 = sc * fmaf(d2, s, w2);
      s *= sc;
    }
    m = cm;
    arg = col0 + ti[0];
  }
  if (tempered && m != -INFINITY) {
    const float b2 = -m * k2;
    float s4[4] = {0.f, 0.f, 0.f, 0.f}, w4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float y2 = fmaf(t[j], k2, b2);
      const float e = exp2f(y2);  // 0 for masked (-inf) columns
      s4[j & 3] += e;
      w4[j & 3] = fmaf(e, e > 0.f ? y2 : 0.f, w4[j & 3]);
    }
    s += (s4[0] + s4[1]) + (s4[2] + s4[3]);
    w2 += (w4[0] + w4[1]) + (w4[2] + w4[3]);
  }
}

template <int BN>
__global__ void __launch_bounds__(kTcThreads, 1) verify_tc_kernel(const __grid_constant__ CUtensorMap tma_x,
                                                                 const __grid_constant__ CUtensorMap tma_w, int H,
                                                                 int n_mt, TcShape sh, EpiArgs ea) {
  extern __shared__ __align__(1024) unsigned char tc_smem_raw[];
  const uint32_t X_BYTES = static_cast<uint32_t>(sh.xr) * BK * 2;
  constexpr uint32_t W_BYTES = BN * BK * 2;
  constexpr uint32_t TMEM_COLS = BN <= 32 ? 32 : BN <= 64 ? 64 : BN <= 128 ? 128 : 256;
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(tc_smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* xsm = smem;                                  // [sx][xr rows x 128 B]
  unsigned char* wsm = smem + sh.sx * X_BYTES;                // [sw][BN rows x 128 B]
  uint64_t* wfull = reinterpret_cast<uint64_t*>(wsm + sh.sw * W_BYTES);
  uint64_t* wempty = wfull + kMaxStages;
  uint64_t* xfull = wempty + kMaxStages;
  uint64_t* xempty = xfull + kMaxStages;
  uint64_t* accb = xempty + kMaxStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accb + 1);
  float* xh = reinterpret_cast<float*>(tmem_slot + 4);        // [5][BM] upper-half row statistics
  __shared__ int s_fail;

  const int tile = blockIdx.x;
  const int m_t = tile % n_mt, n_t = tile / n_mt;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nk = cdiv(H, BK);

  if (threadIdx.x == 0) {
    s_fail = 0;
    for (int s = 0; s < sh.sw; ++s) {
      tc::mbar_init(wfull + s, 1);
      tc::mbar_init(wempty + s, 1);
    }
    for (int s = 0; s < sh.sx; ++s) {
      tc::mbar_init(xfull + s, 1);
      tc::mbar_init(xempty + s, 1);
    }
    tc::mbar_init(accb, 1);
    tc::fence_mbar_init();
    tc::prefetch_tmap(&tma_x);
    tc::prefetch_tmap(&tma_w);
  }
  if (warp == kWarpMma) tc::tmem_alloc(tmem_slot, TMEM_COLS);
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t taddr = *tmem_slot;

  if (warp == kWarpW) {
    // lm_head is a constant input of the step: its stream starts before the
    // wait on the preceding kernel
    if (lane == 0) {
      for (int i = 0; i < nk; ++i) {
        const int s = i % sh.sw;
        const uint32_t ph = (i / sh.sw) & 1;
        if (!tc::mbar_wait(wempty + s, ph ^ 1)) { s_fail = 1; break; }
        tc::mbar_expect_tx(wfull + s, W_BYTES);
        tc::tma_load_2d(smem_u32(wsm + s * W_BYTES), &tma_w, i * BK, n_t * BN, wfull + s);
      }
    }
    __syncwarp();
  } else if (warp == kWarpX) {
    pdl_wait();
    if (lane == 0) {
      for (int i = 0; i < nk; ++i) {
        const int s = i % sh.sx;
        const uint32_t ph = (i / sh.sx) & 1;
        if (!tc::mbar_wait(xempty + s, ph ^ 1)) { s_fail = 1; break; }
        tc::mbar_expect_tx(xfull + s, X_BYTES);
        tc::tma_load_2d(smem_u32(xsm + s * X_BYTES), &tma_x, i * BK, m_t * BM, xfull + s);
      }
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_bf16_f32(BM, BN);
      for (int i = 0; i < nk; ++i) {
        const int sw = i % sh.sw, sx = i % sh.sx;
        if (!tc::mbar_wait(wfull + sw, (i / sh.sw) & 1) || !tc::mbar_wait(xfull + sx, (i / sh.sx) & 1)) {
          s_fail = 1;
          break;
        }
        tc::fence_after_sync();
        const uint32_t sa = smem_u32(xsm + sx * X_BYTES), sb = smem_u32(wsm + sw * W_BYTES);
#pragma unroll
        for (int k = 0; k < BK / 16; ++k)
          tc::mma_bf16(taddr, tc::smem_desc_sw128(sa + k * 32), tc::smem_desc_sw128(sb + k * 32), idesc,
                       (i | k) != 0);
        tc::mma_commit(wempty + sw);
        tc::mma_commit(xempty + sx);
      }
      tc::mma_commit(accb);  // fires once every issued MMA has completed
    }
    __syncwarp();
  } else {
    pdl_wait();
    // ---- epilogue: thread = one tree-node row, one column group of the tile ----
    const int quad = warp & 3, grp = warp >> 2;
    const int row = quad * 32 + lane;
    const int r = m_t * BM + row;
    const bool valid_row = r < ea.R;
    const uint32_t tl = taddr + (static_cast<uint32_t>(quad * 32) << 16);
    const int n0 = n_t * BN;
    const int ncol = min(BN, ea.V - n0);  // valid columns of this tile
    constexpr int NCH = (BN + 31) / 32;
    const int ch0 = grp * NCH / kColGroups, ch1 = (grp + 1) * NCH / kColGroups;
    // While the MMAs run: which of this row's children have their token in
    // this group's columns (bit k: child c_beg + k; a node has < 64 children).
    int b = 0, c_beg = 0;
    uint64_t hits = 0;
    if (valid_row) {
      b = r / ea.T;
      const int node = r % ea.T;
      c_beg = ea.tr.child_start[node];
      const int c_cnt = ea.tr.child_count[node];
      const int32_t* tok = ea.tokens + static_cast<size_t>(b) * ea.T + c_beg;
      const int lo = n0 + ch0 * 32, hi = n0 + min(ncol, ch1 * 32);
      for (int k0 = 0; k0 < c_cnt; k0 += 8) {
        int t[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) t[u] = k0 + u < c_cnt ? tok[k0 + u] : -1;
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (t[u] >= lo && t[u] < hi) hits |= 1ull << (k0 + u);
      }
    }
    const bool ok = tc::mbar_wait(accb, 0);
    tc::fence_after_sync();
    const bool tempered = ea.inv_tau > 0.f;
    const float k2 = ea.inv_tau * kLog2e;
    float m = -INFINITY, s = 0.f, w2 = 0.f;
    int arg = n0 + ch0 * 32;
    bool nan_seen = false;
#pragma unroll 1
    for (int ch = ch0; ch < ch1; ++ch) {
      const int c0 = ch * 32;
      float v[32];
      tc::tmem_ld32(tl + c0, v);
      if (!valid_row || !ok) continue;
      const int nv = min(32, ncol - c0);
      chunk_stats(v, nv, n0 + c0, k2, tempered, m, arg, s, w2, nan_seen);
      if (ea.logits) {
        float* dst = ea.logits + static_cast<size_t>(r) * ea.V + n0 + c0;
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (j < nv) dst[j] = v[j];
      }
      for (uint64_t hm = hits; hm; hm &= hm - 1) {
        const int k = __ffsll(static_cast<long long>(hm)) - 1;
        const int c = c_beg + k;
        const int rel = ea.tokens[static_cast<size_t>(b) * ea.T + c] - (n0 + c0);
        if (rel >= 0 && rel < nv) {
          float z = 0.f;
#pragma unroll
          for (int j = 0; j < 32; ++j) z = (j == rel) ? v[j] : z;
          ea.child_z[static_cast<size_t>(b) * ea.T + c] = z;
        }
      }
    }
    // groups 1.. hand their statistics to group 0, which merges them in
    // column order (ties keep the lower column) and writes the tile's partial
    if (kColGroups > 1) {
      if (grp > 0) {
        float* x = xh + (grp - 1) * 5 * BM;
        x[row] = m;
        x[BM + row] = s;
        x[2 * BM + row] = w2;
        x[3 * BM + row] = __int_as_float(arg);
        x[4 * BM + row] = nan_seen ? 1.f : 0.f;
      }
      asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32) : "memory");
    }
    if (grp == 0 && valid_row) {
      float M = m;
      for (int g = 1; g < kColGroups; ++g) {
        const float mg = xh[(g - 1) * 5 * BM + row];
        if (mg > M) {
          M = mg;
          arg = __float_as_int(xh[(g - 1) * 5 * BM + 3 * BM + row]);
        }
        nan_seen |= xh[(g - 1) * 5 * BM + 4 * BM + row] != 0.f;
      }
      float S = 0.f, W2 = 0.f;
      if (tempered) {
        if (s > 0.f) {
          const float d = (m - M) * k2, sc = exp2f(d);
          S += sc * s;
          W2 += sc * fmaf(d, s, w2);
        }
        for (int g = 1; g < kColGroups; ++g) {
          const float* x = xh + (g - 1) * 5 * BM;
          const float mg = x[row], sg = x[BM + row], wg = x[2 * BM + row];
          if (sg > 0.f) {
            const float d = (mg - M) * k2, sc = exp2f(d);
            S += sc * sg;
            W2 += sc * fmaf(d, sg, wg);
          }
        }
      }
      if (nan_seen) S = __int_as_float(0x7fc00000);
      ea.part[static_cast<size_t>(r) * ea.n_nt + n_t] = make_float4(M, S, W2 * kLn2, __int_as_float(arg));
      if ((!ok || s_fail) && ea.dev_status) atomicOr(ea.dev_status + b, MEDUSA_DEV_TIMEOUT);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == kWarpMma) tc::tmem_dealloc(taddr, TMEM_COLS);
}

// ------------------------------------------------------------------------
// K5, fp32: GEMV logits, then per-(row, tile) statistics.
// ------------------------------------------------------------------------
constexpr int kThreads = 256, kWarps = 8, kRows = 4;

template <int BMAX>
__global__ void __launch_bounds__(kThreads) verify_gemv_f32_kernel(const float* __restrict__ x,
                                                                   const float* __restrict__ lm, int r0, int nb,
                                                                   int H, int V, int groups, float* __restrict__ z) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  float* xs = reinterpret_cast<float*>(smem_raw);
  pdl_wait();
  stage_rows(xs, x + static_cast<size_t>(r0) * H, H, nb, H);
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int g = 0; g < groups; ++g) {
    const long v0 = (static_cast<long>(blockIdx.x) * groups * kWarps + static_cast<long>(g) * kWarps + warp) * kRows;
    if (v0 >= V) break;
    const int valid = V - v0 < kRows ? static_cast<int>(V - v0) : kRows;
    float acc[kRows][BMAX];
    gemv_rows<float, BMAX, kRows, 2>(lm, static_cast<size_t>(v0), valid, H, xs, nb, acc);
#pragma unroll
    for (int rr = 0; rr < kRows; ++rr)
#pragma unroll
      for (int bb = 0; bb < BMAX; ++bb)
        if (rr < valid && bb < nb && lane == ((rr * BMAX + bb) & 31))
          z[static_cast<size_t>(r0 + bb) * V + v0 + rr] = acc[rr][bb];
  }
}

__global__ void __launch_bounds__(256) verify_stats_kernel(const float* __restrict__ z, EpiArgs ea) {
  const int t = blockIdx.x, r = blockIdx.y;
  const int n0 = t * F32_TILE;
  pdl_wait();
  const int col = n0 + threadIdx.x;
  const float v = col < ea.V ? z[static_cast<size_t>(r) * ea.V + col] : -INFINITY;
  __shared__ float sm[8];
  __shared__ int si[8];
  __shared__ float sw[8];
  float m = col < ea.V ? v : -INFINITY;
  int arg = col < ea.V ? col : 0x7fffffff;
  if (m != m) { m = -INFINITY; }
  warp_argmax(m, arg);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) { sm[warp] = m; si[warp] = arg; }
  __syncthreads();
  m = -INFINITY;
  arg = 0x7fffffff;
  for (int i = 0; i < 8; ++i)
    if (better(sm[i], si[i], m, arg)) { m = sm[i]; arg = si[i]; }
  if (arg == 0x7fffffff) arg = n0;
  float s = 0.f, w = 0.f;
  if (col < ea.V && ea.inv_tau > 0.f) {
    const float y = (v - m) * ea.inv_tau;
    s = expf(y);
    w = s * y;
  }
  s = warp_sum(s);
  w = warp_sum(w);
  __syncthreads();
  if (lane == 0) { sm[warp] = s; sw[warp] = w; }
  __syncthreads();
  if (threadIdx.x == 0) {
    float S = 0.f, W = 0.f;
    for (int i = 0; i < 8; ++i) { S += sm[i]; W += sw[i]; }
    ea.part[static_cast<size_t>(r) * ea.n_nt + t] = make_float4(m, S, W, __int_as_float(arg));
  }
  // children whose token lies in this tile
  const int b = r / ea.T, node = r % ea.T;
  const int c_beg = ea.tr.child_start[node], c_cnt = ea.tr.child_count[node];
  for (int c = c_beg + threadIdx.x; c < c_beg + c_cnt; c += blockDim.x) {
    const int tok = ea.tokens[static_cast<size_t>(b) * ea.T + c];
    if (tok >= n0 && tok < n0 + F32_TILE && tok < ea.V) ea.child_z[static_cast<size_t>(b) * ea.T + c] = z[static_cast<size_t>(r) * ea.V + tok];
  }
}

// ------------------------------------------------------------------------
// K6a: merge the per-tile statistics of each node (warp per row, fixed order).
// M = max m_t; S = sum s_t e^{(m_t-M)/tau}; W = sum e^{(m_t-M)/tau} (w_t + s_t (m_t-M)/tau)
// so that with q = softmax(z/tau): H = ln S - W / S.
// ------------------------------------------------------------------------
// One row's tile statistics merged by a warp, tiles in fixed order.
__device__ inline float4 merge_row(const float4* __restrict__ pr, int n_nt, float inv_tau) {
  const int lane = threadIdx.x & 31;
  float m = -INFINITY;
  int arg = 0x7fffffff;
  for (int t = lane; t < n_nt; t += 32) {
    const float4 q = pr[t];
    if (better(q.x, __float_as_int(q.w), m, arg)) { m = q.x; arg = __float_as_int(q.w); }
  }
  warp_argmax(m, arg);
  float S = 0.f, W = 0.f;
  bool nan_seen = false;
  if (inv_tau > 0.f) {
    for (int t = lane; t < n_nt; t += 32) {
      const float4 q = pr[t];
      nan_seen |= q.y != q.y;
      if (q.y > 0.f) {
        const float d = (q.x - m) * inv_tau;
        const float sc = expf(d);
        S = fmaf(q.y, sc, S);
        W = fmaf(sc, fmaf(q.y, d, q.z), W);
      }
    }
    S = warp_sum(S);
    W = warp_sum(W);
  } else {
    for (int t = lane; t < n_nt; t += 32) nan_seen |= pr[t].y != pr[t].y;
  }
  nan_seen = __any_sync(0xffffffffu, nan_seen);
  return make_float4(m, nan_seen ? __int_as_float(0x7fc00000) : S, W, __int_as_float(arg));
}

struct AcceptArgs {
  medusa_tree_dev tr;
  const int32_t* tokens;
  const float4* part;  // [R, n_nt] tile statistics
  int n_nt, R;
  float4* rowst;       // [R] merged statistics
  int* tickets;        // [B] self-resetting
  const float* child_z;
  float inv_tau, thr, alpha;
  float* node_p;
  float* node_H;
  int32_t* accept_len;
  int32_t* best_path;
  int32_t* best_node;
  int32_t* accepted_tokens;
  int32_t* next_root;
  int32_t* dev_status;
};

// ------------------------------------------------------------------------
// K6b: typical acceptance of request b, longest kept prefix, next root
// (whole CTA; the request's merged statistics are in a.rowst).
// ------------------------------------------------------------------------
__device__ void accept_request(const AcceptArgs& a, int b, unsigned char* s_acc, const int16_t* s_par,
                               const int16_t* s_dep, int* s_sc) {
  const medusa_tree_dev& tr = a.tr;
  const int T = tr.T;
  const size_t base = static_cast<size_t>(b) * T;
  int& s_best = s_sc[0];
  int& s_path = s_sc[1];
  int& s_nan = s_sc[2];
  if (threadIdx.x == 0) { s_best = 0; s_path = 0x7fffffff; s_nan = 0; }
  __syncthreads();
  for (int c = threadIdx.x; c < T; c += blockDim.x) {
    const float4 own = __ldcg(a.rowst + base + c);
    if (a.node_H) {
      float H = 0.f;
      if (a.inv_tau > 0.f) H = logf(own.y) - own.z / own.y;
      a.node_H[base + c] = H;
    }
    if (own.x != own.x || own.y != own.y) s_nan = 1;
    if (c == 0) {
      s_acc[0] = 1;
      if (a.node_p) a.node_p[base] = 1.f;
      continue;
    }
    const float4 par = __ldcg(a.rowst + base + s_par[c]);
    const int32_t tok = a.tokens[base + c];
    bool acc;
    float p;
    if (a.inv_tau > 0.f) {
      const float H = logf(par.y) - par.z / par.y;
      p = expf((a.child_z[base + c] - par.x) * a.inv_tau) / par.y;
      acc = p > fminf(a.thr, a.alpha * expf(-H));
    } else {
      acc = tok == __float_as_int(par.w);
      p = acc ? 1.f : 0.f;
    }
    s_acc[c] = acc ? 1 : 0;
    if (a.node_p) a.node_p[base + c] = p;
  }
  __syncthreads();
  for (int d = 1; d <= tr.dmax; ++d) {
    for (int c = threadIdx.x; c < T; c += blockDim.x)
      if (s_dep[c] == d) s_acc[c] = s_acc[c] && s_acc[s_par[c]];
    __syncthreads();
  }
  // deepest kept node, ties to the lowest canonical index
  int key = 0xFFFF;  // root: depth 0, index 0
  for (int c = threadIdx.x; c < T; c += blockDim.x)
    if (s_acc[c]) key = max(key, (static_cast<int>(s_dep[c]) << 16) | (0xFFFF - c));
  for (int o = 16; o > 0; o >>= 1) key = max(key, __shfl_xor_sync(0xffffffffu, key, o));
  if ((threadIdx.x & 31) == 0) atomicMax(&s_best, key);
  __syncthreads();
  const int best = 0xFFFF - (s_best & 0xFFFF);
  for (int p = threadIdx.x; p < tr.P; p += blockDim.x) {
    const int leaf = tr.leaf[p];
    if ((tr.mask[static_cast<size_t>(leaf) * tr.mask_words + best / 32] >> (best % 32)) & 1u) atomicMin(&s_path, p);
  }
  __syncthreads();
  // accepted tokens root..best, read off best's ancestor-mask row
  const int a_len = s_dep[best];
  int32_t* out = a.accepted_tokens + static_cast<size_t>(b) * (tr.dmax + 1);
  for (int t = threadIdx.x; t < T; t += blockDim.x)
    if ((tr.mask[static_cast<size_t>(best) * tr.mask_words + t / 32] >> (t % 32)) & 1u)
      out[s_dep[t]] = a.tokens[base + t];
  for (int d = a_len + 1 + threadIdx.x; d <= tr.dmax; d += blockDim.x) out[d] = -1;
  if (threadIdx.x == 0) {
    a.accept_len[b] = a_len;
    a.best_node[b] = best;
    a.best_path[b] = s_path;
    a.next_root[b] = __float_as_int(__ldcg(a.rowst + base + best).w);
    if (s_nan && a.dev_status) atomicOr(a.dev_status + b, MEDUSA_DEV_NAN);
  }
  __syncthreads();
}

// ------------------------------------------------------------------------
// K6: merge each node's tile statistics (warp per node, kMergeRows nodes per
// CTA, tiles in fixed order); the last CTA to finish a request's nodes
// (ticket per request) then runs that request's acceptance.
// ------------------------------------------------------------------------
constexpr int kMergeRows = 8;

__global__ void __launch_bounds__(kMergeRows * 32) merge_accept_kernel(AcceptArgs a) {
  // shared: parent[T], depth[T] (int16; the tree tables are constant, so they are
  // read before the wait on the preceding kernel), then acc[T] bytes
  extern __shared__ __align__(16) unsigned char accept_smem[];
  const int T = a.tr.T;
  int16_t* s_par = reinterpret_cast<int16_t*>(accept_smem);
  int16_t* s_dep = s_par + T;
  unsigned char* s_acc = reinterpret_cast<unsigned char*>(s_dep + T);
  __shared__ int s_sc[3];
  __shared__ int s_last;
  for (int c = threadIdx.x; c < T; c += blockDim.x) {
    s_par[c] = static_cast<int16_t>(a.tr.parent[c]);
    s_dep[c] = static_cast<int16_t>(a.tr.depth[c]);
  }
  pdl_wait();
  pdl_trigger();
  const int r0 = blockIdx.x * kMergeRows, r1 = min(a.R, r0 + kMergeRows);
  const int r = r0 + (threadIdx.x >> 5);
  if (r < r1) {
    const float4 v = merge_row(a.part + static_cast<size_t>(r) * a.n_nt, a.n_nt, a.inv_tau);
    if ((threadIdx.x & 31) == 0) a.rowst[r] = v;
  }
  __threadfence();
  __syncthreads();
  for (int b = r0 / T; b <= (r1 - 1) / T; ++b) {
    const int need = ((b + 1) * T - 1) / kMergeRows - (b * T) / kMergeRows + 1;  // CTAs holding b's nodes
    if (threadIdx.x == 0) s_last = atomicAdd(a.tickets + b, 1) == need - 1;
    __syncthreads();
    if (s_last) {
      __threadfence();
      accept_request(a, b, s_acc, s_par, s_dep, s_sc);
      if (threadIdx.x == 0) a.tickets[b] = 0;  // ready for the next launch
    }
    __syncthreads();
  }
}

constexpr size_t kTcSmemMax = 227 * 1024 - 1024;  // the kernel's static shared memory takes 1 KB
constexpr size_t kTcFixedBytes = 1024 + (4 * kMaxStages + 1) * 8 + 16 + kHalfXchgBytes;

TcShape tc_shape(const VerifyPlan& p) {
  TcShape sh{};
  sh.BN = p.BN;
  const int rows = p.n_mt == 1 ? p.R : BM;
  sh.xr = std::min(BM, cdiv(rows, 8) * 8);
  const size_t xb = static_cast<size_t>(sh.xr) * BK * 2, wb = static_cast<size_t>(p.BN) * BK * 2;
  sh.sx = 4;
  sh.sw = static_cast<int>(std::min<size_t>(kMaxStages, (kTcSmemMax - kTcFixedBytes - sh.sx * xb) / wb));
  return sh;
}

size_t tc_smem_bytes(const TcShape& sh) {
  return kTcFixedBytes + static_cast<size_t>(sh.sx) * sh.xr * BK * 2 + static_cast<size_t>(sh.sw) * sh.BN * BK * 2;
}

template <int BN>
int launch_tc(const VerifyPlan& p, const CUtensorMap& mx, const CUtensorMap& mw, int H, const EpiArgs& ea,
              cudaStream_t st) {
  const TcShape sh = tc_shape(p);
  if (sh.sw < 2) return MEDUSA_ERR_UNSUPPORTED;
  const size_t smem = tc_smem_bytes(sh);
  auto k = verify_tc_kernel<BN>;
  if (!ensure_dyn_smem(k, smem))
    return MEDUSA_ERR_CUDA;
  if (launch_pdl(k, dim3(p.n_mt * p.n_nt), dim3(kTcThreads), smem, st, mx, mw, H, p.n_mt, sh, ea) != cudaSuccess) {
    (void)cudaGetLastError();
    return MEDUSA_ERR_CUDA;
  }
  MEDUSA_LAUNCH_CHECK();
  return MEDUSA_OK;
}

int dispatch_tc(const VerifyPlan& p, const CUtensorMap& mx, const CUtensorMap& mw, int H, const EpiArgs& ea,
                cudaStream_t st) {
  switch (p.BN) {
#define MEDUSA_BN(n) case n: return launch_tc<n>(p, mx, mw, H, ea, st);
    MEDUSA_BN(16) MEDUSA_BN(32) MEDUSA_BN(48) MEDUSA_BN(64) MEDUSA_BN(80) MEDUSA_BN(96) MEDUSA_BN(112)
    MEDUSA_BN(128) MEDUSA_BN(144) MEDUSA_BN(160) MEDUSA_BN(176) MEDUSA_BN(192) MEDUSA_BN(208) MEDUSA_BN(224)
    MEDUSA_BN(240) MEDUSA_BN(256)
#undef MEDUSA_BN
    default: return MEDUSA_ERR_UNSUPPORTED;
  }
}

}  // namespace

MEDUSA_API size_t medusa_verify_accept_workspace_size(const medusa_tree* tree, int32_t B, int32_t H, int32_t V,
                                                      medusa_dtype dtype) {
  if (!tree || B < 1 || H < 1 || V < 1) return 0;
  VerifyPlan p = plan_verify(B, tree->T, V, dtype);
  return carve_verify_ws(nullptr, p, V, dtype).bytes;
}

MEDUSA_API int medusa_verify_accept(const medusa_tree* tree, const void* x, const void* lm_head,
                                    const int32_t* tree_tokens, int32_t B, int32_t H, int32_t V, medusa_dtype dtype,
                                    float temperature, float posterior_threshold, float posterior_alpha,
                                    float* logits, float* node_p, float* node_H, int32_t* accept_len,
                                    int32_t* best_path, int32_t* best_node, int32_t* accepted_tokens,
                                    int32_t* next_root, int32_t* dev_status, void* ws, size_t ws_bytes,
                                    medusa_stream_t stream) {
  if (!tree || !x || !lm_head || !tree_tokens || !accept_len || !best_path || !best_node || !accepted_tokens ||
      !next_root)
    return MEDUSA_ERR_INVALID_ARG;
  if (B < 1 || B > MEDUSA_MAX_BATCH || H < 8 || V < 1 || !(temperature >= 0.f)) return MEDUSA_ERR_INVALID_ARG;
  if (dtype != MEDUSA_F32 && dtype != MEDUSA_BF16) return MEDUSA_ERR_INVALID_ARG;
  if (H % 8 != 0) return MEDUSA_ERR_UNSUPPORTED;
  const void* ptrs[] = {x, lm_head, tree_tokens, accept_len, best_path, best_node, accepted_tokens, next_root};
  for (const void* q : ptrs)
    if (!aligned16(q)) return MEDUSA_ERR_ALIGNMENT;
  const void* opt[] = {logits, node_p, node_H, dev_status, ws};
  for (const void* q : opt)
    if (q && !aligned16(q)) return MEDUSA_ERR_ALIGNMENT;
  const int T = tree->T;
  VerifyPlan p = plan_verify(B, T, V, dtype);
  VerifyWs w = carve_verify_ws(ws, p, V, dtype);
  if (!ws || ws_bytes < w.bytes) return MEDUSA_ERR_WORKSPACE;
  auto st = reinterpret_cast<cudaStream_t>(stream);
  const float inv_tau = temperature > 0.f ? 1.f / temperature : 0.f;
  EpiArgs ea{p.R, V, T, p.n_nt, tree_tokens, tree->dev, inv_tau, logits, w.part, w.child_z, dev_status};

  if (dtype == MEDUSA_BF16) {
    CUtensorMap mx, mw;
    if (!make_tmap_bf16(&mx, x, p.R, H, tc_shape(p).xr) || !make_tmap_bf16(&mw, lm_head, V, H, p.BN))
      return MEDUSA_ERR_CUDA;
    const int rc = dispatch_tc(p, mx, mw, H, ea, st);
    if (rc != MEDUSA_OK) return rc;
  } else {
    float* z = logits ? logits : w.zbuf;
    ea.logits = nullptr;
    const int rows_per_launch = 16;
    const long vrows = V;
    const int groups = std::max(1L, (vrows + 148L * 4 * kWarps * kRows - 1) / (148L * 4 * kWarps * kRows));
    const int ctas = cdiv(V, groups * kWarps * kRows);
    for (int r0 = 0; r0 < p.R; r0 += rows_per_launch) {
      const int nb = std::min(rows_per_launch, p.R - r0);
      const size_t smem = static_cast<size_t>(nb) * H * 4;
      if (smem > 200 * 1024) return MEDUSA_ERR_UNSUPPORTED;
      auto k = nb <= 4 ? verify_gemv_f32_kernel<4> : nb <= 8 ? verify_gemv_f32_kernel<8> : verify_gemv_f32_kernel<16>;
      if (!ensure_dyn_smem(k, smem))
        return MEDUSA_ERR_CUDA;
      if (launch_pdl(k, dim3(ctas), dim3(kThreads), smem, st, static_cast<const float*>(x),
                     static_cast<const float*>(lm_head), r0, nb, H, V, groups, z) != cudaSuccess) {
        (void)cudaGetLastError();
        return MEDUSA_ERR_CUDA;
      }
      MEDUSA_LAUNCH_CHECK();
    }
    if (launch_pdl(verify_stats_kernel, dim3(p.n_nt, p.R), dim3(256), 0, st, static_cast<const float*>(z), ea) !=
        cudaSuccess) {
      (void)cudaGetLastError();
      return MEDUSA_ERR_CUDA;
    }
    MEDUSA_LAUNCH_CHECK();
  }
  AcceptArgs aa{tree->dev, tree_tokens, w.part, p.n_nt, p.R, w.rowst, w.tickets, w.child_z, inv_tau,
                posterior_threshold, posterior_alpha, node_p, node_H, accept_len, best_path, best_node,
                accepted_tokens, next_root, dev_status};
  if (launch_pdl(merge_accept_kernel, dim3(cdiv(p.R, kMergeRows)), dim3(kMergeRows * 32), static_cast<size_t>(T) * 5,
                 st, aa) != cudaSuccess) {
    (void)cudaGetLastError();
    return MEDUSA_ERR_CUDA;
  }
  MEDUSA_LAUNCH_CHECK();
  return MEDUSA_OK;
}
