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
// rows (B*T) and N = vocabulary.  A persistent kernel: tcgen05.mma accumulates
// 128 x BN tiles in two alternating TMEM accumulators from TMA-fed,
// 128-byte-swizzled shared-memory rings (one producer thread per operand, one
// MMA thread).  The epilogue (eight warps, one TMEM lane = one tree node) never
// writes the logits unless asked: it reduces its vocabulary tile to (max,
// argmax, sum of exp, sum of exp * logit) at the temperature and picks out the
// logits of the node's children tokens.  The same kernel, with a logits-only
// epilogue and several GEMMs per launch, serves the Medusa heads at larger
// batches (launch_group_logits_bf16).
// K5 (fp32): CUDA-core GEMV into a logits buffer, then the same statistics.
// K6 merges the statistics of every node and tests its children; the last CTA
// of a request then picks the longest kept prefix and the next root.
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
  int qr, n_g, n_tiles, grid;  // bf16: rows per TMEM lane quadrant, groups, tiles, persistent CTAs
  int n_parts;            // statistics partials per row (bf16, one row tile: one per CTA)
};

// bf16: the row tiles split the B*T rows evenly (4*qr <= 128 rows each).  With
// one row tile the GEMM streams lm_head once: BN minimises what the busiest
// CTA loads, its lm_head rows plus the tree rows X again for every tile (X
// rows cost about twice a weight row: every CTA requests the same lines), and
// a little for the last tile's exposed epilogue.  At the 7B vocabulary that
// is one 224-column tile per CTA.  With several row tiles the GEMM is
// compute-bound and takes the widest MMA.
// tcgen05 GEMM plan for R rows, n_g groups and V columns per group.
VerifyPlan plan_tc(int R, int n_g, int V, bool topk = false) {
  VerifyPlan p{};
  p.R = R;
  const int sms = device_sm_count();
  p.n_mt = cdiv(R, BM);
  p.qr = cdiv(R, 4 * p.n_mt);
  if (p.n_mt == 1) {
    long best = -1;
    // the top-k epilogue is built for tile widths 128..256 in steps of 32
    for (int bn = topk ? 128 : 16; bn <= 256; bn += topk ? 32 : 16) {
      const long per_cta = cdiv(n_g * cdiv(V, bn), sms);
      const long cost = 8 * per_cta * (bn + 8 * p.qr) + bn;
      if (best < 0 || cost <= best) {
        best = cost;
        p.BN = bn;
      }
    }
  } else {
    p.BN = 256;
  }
  p.n_nt = cdiv(V, p.BN);
  p.n_g = n_g;
  p.n_tiles = n_g * p.n_mt * p.n_nt;
  p.grid = std::min(p.n_tiles, sms);
  p.n_parts = p.n_mt == 1 ? p.grid : p.n_nt;
  return p;
}

VerifyPlan plan_verify(int B, int T, int V, medusa_dtype dt) {
  if (dt == MEDUSA_BF16) return plan_tc(B * T, 1, V);
  VerifyPlan p{};
  p.R = B * T;
  p.n_mt = 1;
  p.n_g = 1;
  p.BN = F32_TILE;
  p.n_nt = cdiv(V, F32_TILE);
  p.n_parts = p.n_nt;
  return p;
}

struct VerifyWs {
  float4* part;      // [R, n_parts] (max, sum exp, sum exp*y, argmax bits)
  float* child_z;    // [R] logit of node c's token under its parent (indexed by c)
  float4* rowst;     // [R] merged statistics
  unsigned char* acc;  // [R] each node's acceptance test against its parent
  float* logp;       // [R] ln p of each node under its parent (joint-probability tie-break)
  int* tickets;      // [B] CTAs done with a request's nodes (self-resetting)
  float* zbuf;       // fp32 path: [R, V] logits when the caller gives none
  size_t bytes;
};

VerifyWs carve_verify_ws(void* base, const VerifyPlan& p, int V, medusa_dtype dt) {
  VerifyWs w{};
  size_t o = 0;
  auto take = [&](size_t n) { size_t s = o; o = align_up(o + n, 256); return s; };
  size_t op = take(static_cast<size_t>(p.R) * p.n_parts * 16), oc = take(static_cast<size_t>(p.R) * 4),
         orow = take(static_cast<size_t>(p.R) * 16), otk = take(static_cast<size_t>(p.R) * 4),
         oa = take(static_cast<size_t>(p.R)), olp = take(static_cast<size_t>(p.R) * 4);
  size_t oz = dt == MEDUSA_F32 ? take(static_cast<size_t>(p.R) * V * 4) : 0;
  char* c = static_cast<char*>(base);
  if (c) {
    w.part = reinterpret_cast<float4*>(c + op);
    w.child_z = reinterpret_cast<float*>(c + oc);
    w.rowst = reinterpret_cast<float4*>(c + orow);
    w.tickets = reinterpret_cast<int*>(c + otk);
    w.acc = reinterpret_cast<unsigned char*>(c + oa);
    w.logp = reinterpret_cast<float*>(c + olp);
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
  float4* part;      // null: logits only (no statistics, no child gathers)
  float* child_z;
  int32_t* dev_status;
  int n_g;           // GEMMs in the launch (group g: weight rows g*V.., activation group g)
  int topk_k;        // top-k epilogue: candidates [rows][n_g][n_nt][topk_k] of each (row, group, vocabulary tile)
  float* cand_v;
  int* cand_i;
};

constexpr int kEpiTopkMax = 16;  // most candidates the top-k epilogue keeps per (row, tile)

// ------------------------------------------------------------------------
// K5, bf16: persistent tcgen05 GEMM with the statistics epilogue.
// A tile is 4*qr tree rows x BN vocabulary columns; CTA c takes tiles c,
// c + grid, ...  Warps 0..kEpiWarps-1 run the epilogue (warp w reads TMEM
// lanes 32*(w%4).. and the (w/4)-th of kEpiWarps/4 column groups); the next
// warp streams lm_head tiles, the next issues the MMAs and owns TMEM, the last
// streams the tree rows X.  Two TMEM accumulators alternate between tiles, so
// the epilogue of one tile runs under the MMAs of the next.
// A tile's rows are spread over the four TMEM lane quadrants (qr <= 32 rows
// each: quadrant q of row tile m holds rows m*4*qr + q*qr ..), so that small
// trees keep every epilogue warp busy; X stages are 128 rows (four TMA boxes
// of qr rows at shared-memory rows 0, 32, 64, 96; rows past a box are never
// written and feed only accumulator rows that are never read).
// lm_head (from HBM) and X (from L2, shared by every CTA) run in separate
// rings: a deep one for the weight stream, a shallow one for X.
// ------------------------------------------------------------------------
constexpr int kMaxStagesW = 16;
constexpr int kMaxStagesX = 4;
constexpr uint32_t kXStageBytes = BM * BK * 2;
constexpr int kEpiWarps = 8;
constexpr int kWarpW = kEpiWarps, kWarpMma = kEpiWarps + 1, kWarpX = kEpiWarps + 2;
constexpr int kTcThreads = (kEpiWarps + 3) * 32;
constexpr int kColGroups = kEpiWarps / 4;
constexpr size_t kXchgBytes = 2 * (kColGroups - 1) * BM * 5 * 4;  // per-row statistics of groups 1.., 2 buffers
constexpr size_t kTopkBufBytes = kEpiWarps * 64 * 4;  // top-k epilogue: one 64-column row buffer per warp

struct TcShape {
  int BN;       // vocabulary columns per tile
  int qr;       // tree rows per TMEM lane quadrant (a row tile holds 4*qr rows)
  int n_mt;     // row tiles
  int n_nt;     // vocabulary tiles per group
  int n_g;      // groups (independent GEMMs sharing the launch)
  int n_tiles;  // n_g * n_nt * n_mt; tile t is row tile t % n_mt, then vocabulary tile, then group
  int sw;       // lm_head ring stages
  int sx;       // X ring stages (<= kMaxStagesX)
  int topk;     // top-k epilogue (its exchange buffer follows the statistics one)
};

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Running statistics of one row over a block of NCH*16 columns v[0..nv):
// maximum and its first column (tree reduction per 16 columns, then the
// chunks in column order), then, at temperature > 0, the sums s = sum 2^y2
// and w2 = sum 2^y2 * y2 with y2 = (z - m) * k2, k2 = log2(e) / temperature,
// rescaled when the maximum grows.  NaN never wins the maximum.
template <int NCH>
__device__ inline void block_stats(float (&v)[NCH * 16], int nv, int col0, float k2, bool tempered, float& m,
                                   int& arg, float& s, float& w2, bool& nan_seen) {
  constexpr int N = NCH * 16;
#pragma unroll
  for (int j = 0; j < N; ++j) {
    const bool in = j < nv;
    nan_seen |= in && v[j] != v[j];
    v[j] = (in && v[j] == v[j]) ? v[j] : -INFINITY;
  }
  float bm = -INFINITY;
  int bi = 0;
#pragma unroll
  for (int c = 0; c < NCH; ++c) {
    float tv[8];
    int ti[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const bool take = v[c * 16 + j + 8] > v[c * 16 + j];
      tv[j] = take ? v[c * 16 + j + 8] : v[c * 16 + j];
      ti[j] = take ? j + 8 : j;
    }
#pragma unroll
    for (int h = 4; h >= 1; h >>= 1) {
#pragma unroll
      for (int j = 0; j < h; ++j) {
        const bool take = tv[j + h] > tv[j];
        tv[j] = take ? tv[j + h] : tv[j];
        ti[j] = take ? ti[j + h] : ti[j];
      }
    }
    if (tv[0] > bm) {
      bm = tv[0];
      bi = c * 16 + ti[0];
    }
  }
  if (bm > m) {
    if (tempered && s > 0.f) {
      const float d2 = (m - bm) * k2;
      const float sc = ex2_approx(d2);
      w2 = sc * fmaf(d2, s, w2);
      s *= sc;
    }
    m = bm;
    arg = col0 + bi;
  }
  if (tempered && m != -INFINITY) {
    const float b2 = -m * k2;
    float s4[4] = {0.f, 0.f, 0.f, 0.f}, w4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < N; ++j) {
      const float y2 = fmaf(v[j], k2, b2);
      const float e = ex2_approx(y2);  // 0 for masked (-inf) columns
      s4[j & 3] += e;
      w4[j & 3] = fmaf(e, e > 0.f ? y2 : 0.f, w4[j & 3]);
    }
    s += (s4[0] + s4[1]) + (s4[2] + s4[3]);
    w2 += (w4[0] + w4[1]) + (w4[2] + w4[3]);
  }
}

// One block of NCH 16-column chunks starting at chunk `ch` of the accumulator
// at `tl`: load, statistics, logits copy and child gathers.
template <int NCH>
__device__ inline void epi_block(const EpiArgs& ea, uint32_t tl, int ch, int ncol, int n0, int r, int g, int b,
                                 bool use, bool stats, float k2, bool tempered, int c_beg, uint64_t hits, float& m,
                                 int& arg, float& s, float& w2, bool& nan_seen) {
  float v[NCH * 16];
  tc::tmem_ld16n<NCH>(tl + ch * 16, v);
  if (!use) return;
  const int c0 = ch * 16;
  const int nv = min(NCH * 16, ncol - c0);
  if (ea.logits && nv > 0) {
    float* dst = ea.logits + (static_cast<size_t>(r) * ea.n_g + g) * ea.V + n0 + c0;
#pragma unroll
    for (int j = 0; j < NCH * 16; ++j)
      if (j < nv) dst[j] = v[j];
  }
  for (uint64_t hm = hits; hm; hm &= hm - 1) {
    const int k = __ffsll(static_cast<long long>(hm)) - 1;
    const int c = c_beg + k;
    const int rel = ea.tokens[static_cast<size_t>(b) * ea.T + c] - (n0 + c0);
    if (rel >= 0 && rel < nv) {
      float z = 0.f;
#pragma unroll
      for (int j = 0; j < NCH * 16; ++j) z = (j == rel) ? v[j] : z;
      ea.child_z[static_cast<size_t>(b) * ea.T + c] = z;
    }
  }
  if (stats) block_stats<NCH>(v, nv, n0 + c0, k2, tempered, m, arg, s, w2, nan_seen);
}

__device__ inline bool failed(const volatile int* f) { return *f != 0; }

// Top-k epilogue of one accumulator tile for the rows in `rows` (bits = lanes
// of this warp's quadrant).  Per row: its columns go through `buf` (one lane
// stores 64 columns, all lanes read two), so the row's top-k is a list spread
// over lanes 0..k-1 (value descending, equal values by the lower column) and a
// column enters only if it beats the k-th entry: a ballot finds such columns,
// each insertion counts the entries ahead of it and shifts the rest down one
// lane.  NaN never enters.  The row's k entries go to the candidate buffer
// (unfilled ones as NaN / -1), and its logits to ea.logits when that is given.
template <int BN>
__device__ __forceinline__ void topk_tile(const EpiArgs& ea, uint32_t tl, int ncol, int n0, int r_lane, int g, int n_t,
                                       uint32_t rows, float* buf) {
  constexpr int NCH = BN / 16;  // a multiple of 2: loads of 4 chunks, then possibly one of 2
  const int lane = threadIdx.x & 31, k = ea.topk_k;
  for (; rows; rows &= rows - 1) {
    const int rr = __ffs(rows) - 1;
    const int r = __shfl_sync(0xffffffffu, r_lane, rr);
    float* zrow = ea.logits ? ea.logits + (static_cast<size_t>(r) * ea.n_g + g) * ea.V + n0 : nullptr;
    float lv = -INFINITY, tv = -INFINITY;  // lane j < k: entry j; tv/ti: entry k-1
    int li = 0x7fffffff, ti = 0x7fffffff;
#pragma unroll 1
    for (int ch = 0; ch < NCH; ch += 4) {
      float v[64];
      int nc = 4;
      if (NCH - ch >= 4) {
        tc::tmem_ld16n<4>(tl + ch * 16, v);
      } else {
        tc::tmem_ld16n<2>(tl + ch * 16, *reinterpret_cast<float(*)[32]>(v));
        nc = 2;
      }
      if (lane == rr) {
#pragma unroll
        for (int q = 0; q < 16; ++q)
          if (q < nc * 4) *reinterpret_cast<float4*>(buf + 4 * q) = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
      }
      __syncwarp();
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int c = ch * 16 + h * 32 + lane;
        const bool in = h * 32 < nc * 16 && c < ncol;
        const float x = in ? buf[h * 32 + lane] : __int_as_float(0x7fc00000);
        const int id = n0 + c;
        if (zrow && in) zrow[c] = x;
        uint32_t cand = __ballot_sync(0xffffffffu, better(x, id, tv, ti));
        while (cand) {
          const int src = __ffs(cand) - 1;
          const float xv = __shfl_sync(0xffffffffu, x, src);
          const int xi = __shfl_sync(0xffffffffu, id, src);
          // x beats entry k-1, so fewer than k entries are ahead of it
          const int pos = __popc(__ballot_sync(0xffffffffu, lane < k && better(lv, li, xv, xi)));
          const float uv = __shfl_up_sync(0xffffffffu, lv, 1);
          const int ui = __shfl_up_sync(0xffffffffu, li, 1);
          if (lane == pos) {
            lv = xv;
            li = xi;
          } else if (lane > pos && lane < k) {
            lv = uv;
            li = ui;
          }
          tv = __shfl_sync(0xffffffffu, lv, k - 1);
          ti = __shfl_sync(0xffffffffu, li, k - 1);
          cand &= cand - 1;
          cand &= __ballot_sync(0xffffffffu, better(x, id, tv, ti));
        }
      }
      __syncwarp();
    }
    if (lane < k) {
      const size_t o = ((static_cast<size_t>(r) * ea.n_g + g) * ea.n_nt + n_t) * k + lane;
      const bool filled = li != 0x7fffffff;
      ea.cand_v[o] = filled ? lv : __int_as_float(0x7fc00000);
      ea.cand_i[o] = filled ? li : -1;
    }
  }
}

template <int BN, bool TOPK>
__global__ void __launch_bounds__(kTcThreads, 1) verify_tc_kernel(const __grid_constant__ CUtensorMap tma_x,
                                                                 const __grid_constant__ CUtensorMap tma_w, int H,
                                                                 TcShape sh, EpiArgs ea) {
  extern __shared__ __align__(1024) unsigned char tc_smem_raw[];
  constexpr uint32_t W_BYTES = BN * BK * 2;
  constexpr int ACC_STRIDE = (BN + 31) / 32 * 32;  // TMEM columns from one accumulator to the other
  constexpr uint32_t TMEM_COLS = 2 * ACC_STRIDE <= 64 ? 64 : 2 * ACC_STRIDE <= 128 ? 128 : 2 * ACC_STRIDE <= 256 ? 256 : 512;
  constexpr int NCH = BN / 16;  // 16-column chunks of a tile
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(tc_smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* xsm = smem;                             // [sx][128 rows x 128 B]
  unsigned char* wsm = smem + sh.sx * kXStageBytes;      // [sw][BN rows x 128 B]
  uint64_t* wfull = reinterpret_cast<uint64_t*>(wsm + sh.sw * W_BYTES);
  uint64_t* wempty = wfull + kMaxStagesW;
  uint64_t* xfull = wempty + kMaxStagesW;
  uint64_t* xempty = xfull + kMaxStagesX;
  uint64_t* acc_full = xempty + kMaxStagesX;
  uint64_t* acc_empty = acc_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);
  float* xh = reinterpret_cast<float*>(tmem_slot + 4);  // [2][kColGroups-1][5][BM] statistics of groups 1..
  float* tbuf = xh + kXchgBytes / 4;  // top-k epilogue: [kEpiWarps][64] one row's columns
  __shared__ int s_fail;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nk = cdiv(H, BK);
  const int qr = sh.qr;
  // In the memory-bound GEMM (one row tile) the K loop of vocabulary tile n_t
  // starts at block n_t * nk / n_nt, so the CTAs streaming at the same time
  // spread their requests over more DRAM pages; the rotation depends on the
  // column tile only, so every group of a grouped GEMM sums a column in the
  // same order (equal groups give bit-identical results).  The compute-bound
  // GEMM keeps the CTAs that share a weight tile in step, so the tile is still
  // in L2 for all of them.
  auto rot_of = [&](int t) {
    return sh.n_mt == 1 ? static_cast<int>((static_cast<long>((t / sh.n_mt) % sh.n_nt) * nk) / sh.n_nt) : 0;
  };

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
    for (int a = 0; a < 2; ++a) {
      tc::mbar_init(acc_full + a, 1);
      tc::mbar_init(acc_empty + a, kEpiWarps);
    }
    tc::fence_mbar_init();
    tc::prefetch_tmap(&tma_x);
    tc::prefetch_tmap(&tma_w);
  }
  if (warp == kWarpMma) tc::tmem_alloc(tmem_slot, TMEM_COLS);
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t taddr = *tmem_slot;
  pdl_trigger();  // the merge kernel may take its place early (it waits for this grid)

  if (warp == kWarpW) {
    // lm_head is a constant input of the step: its stream starts before the
    // wait on the preceding kernel
    if (lane == 0) {
      int i = 0;
      bool run = true;
      for (int t = blockIdx.x; t < sh.n_tiles && run; t += gridDim.x) {
        const int rest = t / sh.n_mt;
        const int wrow = (rest / sh.n_nt) * ea.V + (rest % sh.n_nt) * BN;  // group g's rows start at g*V
        const int rot = rot_of(t);
        for (int k = 0; k < nk; ++k, ++i) {
          const int s = i % sh.sw;
          if (failed(&s_fail) || !tc::mbar_wait(wempty + s, ((i / sh.sw) & 1) ^ 1)) { s_fail = 1; run = false; break; }
          tc::mbar_expect_tx(wfull + s, W_BYTES);
          tc::tma_load_2d(smem_u32(wsm + s * W_BYTES), &tma_w, ((k + rot) % nk) * BK, wrow, wfull + s);
        }
      }
    }
    __syncwarp();
  } else if (warp == kWarpX) {
    pdl_wait();
    if (lane == 0) {
      int i = 0;
      bool run = true;
      for (int t = blockIdx.x; t < sh.n_tiles && run; t += gridDim.x) {
        const int row0 = (t % sh.n_mt) * 4 * qr;
        const int g = t / sh.n_mt / sh.n_nt;
        const int rot = rot_of(t);
        for (int k = 0; k < nk; ++k, ++i) {
          const int s = i % sh.sx;
          if (failed(&s_fail) || !tc::mbar_wait(xempty + s, ((i / sh.sx) & 1) ^ 1)) { s_fail = 1; run = false; break; }
          tc::mbar_expect_tx(xfull + s, 4u * qr * BK * 2);
          const int kx = ((k + rot) % nk) * BK;
          for (int q = 0; q < 4; ++q) {
            const uint32_t dst = smem_u32(xsm + s * kXStageBytes + q * 32 * BK * 2);
            if (sh.n_g == 1)
              tc::tma_load_2d(dst, &tma_x, kx, row0 + q * qr, xfull + s);
            else  // [rows][groups][H]: box of qr rows of group g
              tc::tma_load_3d(dst, &tma_x, kx, g, row0 + q * qr, xfull + s);
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_bf16_f32(BM, BN);
      // base descriptors of the rings, stepped with desc_add, and running stage
      // and parity counters: the integer work between MMAs bounds their issue rate
      const uint64_t da0 = tc::smem_desc_sw128(smem_u32(xsm)), db0 = tc::smem_desc_sw128(smem_u32(wsm));
      int sw = 0, sx = 0;
      uint32_t pw = 0, px = 0;
      int jl = 0;
      bool run = true;
      for (int t = blockIdx.x; t < sh.n_tiles && run; t += gridDim.x, ++jl) {
        const int a = jl & 1;
        if (failed(&s_fail) || !tc::mbar_wait(acc_empty + a, ((jl >> 1) & 1) ^ 1)) { s_fail = 1; break; }
        tc::fence_after_sync();
        const uint32_t d = taddr + a * ACC_STRIDE;
        for (int k = 0; k < nk; ++k) {
          if (failed(&s_fail) || !tc::mbar_wait(wfull + sw, pw) || !tc::mbar_wait(xfull + sx, px)) {
            s_fail = 1;
            run = false;
            break;
          }
          tc::fence_after_sync();
          const uint64_t da = tc::desc_add(da0, sx * kXStageBytes), db = tc::desc_add(db0, sw * W_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            tc::mma_bf16(d, tc::desc_add(da, kk * 32), tc::desc_add(db, kk * 32), idesc, (k | kk) != 0);
          tc::mma_commit(wempty + sw);
          tc::mma_commit(xempty + sx);
          if (++sw == sh.sw) { sw = 0; pw ^= 1; }
          if (++sx == sh.sx) { sx = 0; px ^= 1; }
        }
        if (run) tc::mma_commit(acc_full + a);  // fires once every MMA of the tile has completed
      }
    }
    __syncwarp();
  } else {
    pdl_wait();
    // ---- epilogue: thread = one tree row (lane < qr) of its quadrant, one column group ----
    const int quad = warp & 3, grp = warp >> 2;
    const int ch0 = grp * NCH / kColGroups, ch1 = (grp + 1) * NCH / kColGroups;
    const bool tempered = ea.inv_tau > 0.f;
    const bool stats = ea.part != nullptr;
    const float k2 = ea.inv_tau * kLog2e;
    int jl = 0;
    bool ok = true;
    float run_m = -INFINITY, run_s = 0.f, run_w2 = 0.f;  // this CTA's tiles folded (one row tile)
    int run_arg = 0x7fffffff;
    bool run_nan = false;
    for (int t = blockIdx.x; t < sh.n_tiles; t += gridDim.x, ++jl) {
      const int a = jl & 1;
      const int m_t = t % sh.n_mt, n_t = (t / sh.n_mt) % sh.n_nt, g = t / sh.n_mt / sh.n_nt;
      const int r = m_t * 4 * qr + quad * qr + lane;
      const bool valid_row = lane < qr && r < ea.R;
      const uint32_t tl = taddr + (static_cast<uint32_t>(quad * 32) << 16) + a * ACC_STRIDE;
      const int n0 = n_t * BN;
      const int ncol = min(BN, ea.V - n0);  // valid columns of this tile
      // While the MMAs run: which of this row's children have their token in
      // this group's columns (bit k: child c_beg + k; a node has < 64 children).
      int b = 0, c_beg = 0;
      uint64_t hits = 0;
      if (valid_row && stats) {
        b = r / ea.T;
        const int node = r % ea.T;
        c_beg = ea.tr.child_start[node];
        const int c_cnt = ea.tr.child_count[node];
        const int32_t* tok = ea.tokens + static_cast<size_t>(b) * ea.T + c_beg;
        const int lo = n0 + ch0 * 16, hi = n0 + min(ncol, ch1 * 16);
        for (int k0 = 0; k0 < c_cnt; k0 += 8) {
          int tk[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) tk[u] = k0 + u < c_cnt ? tok[k0 + u] : -1;
#pragma unroll
          for (int u = 0; u < 8; ++u)
            if (tk[u] >= lo && tk[u] < hi) hits |= 1ull << (k0 + u);
        }
      }
      ok = ok && __all_sync(0xffffffffu, !failed(&s_fail) && tc::mbar_wait(acc_full + a, (jl >> 1) & 1));
      tc::fence_after_sync();
      if constexpr (TOPK) {
        // the two warps of a lane quadrant split its rows by parity; each takes
        // its rows' whole tile, one row at a time, across its 32 lanes
        const uint32_t mine = __ballot_sync(0xffffffffu, valid_row) & (grp ? 0xaaaaaaaau : 0x55555555u);
        if (ok && mine) topk_tile<BN>(ea, tl, ncol, n0, r, g, n_t, mine, tbuf + warp * 64);
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(acc_empty + a);
        continue;
      }
      float m = -INFINITY, s = 0.f, w2 = 0.f;
      int arg = n0 + ch0 * 16;
      bool nan_seen = false;
      if (ok) {
        const bool use = valid_row;
        for (int ch = ch0; ch < ch1; ch += 4) {
          switch (min(4, ch1 - ch)) {
            case 4: epi_block<4>(ea, tl, ch, ncol, n0, r, g, b, use, stats, k2, tempered, c_beg, hits, m, arg, s, w2, nan_seen); break;
            case 3: epi_block<3>(ea, tl, ch, ncol, n0, r, g, b, use, stats, k2, tempered, c_beg, hits, m, arg, s, w2, nan_seen); break;
            case 2: epi_block<2>(ea, tl, ch, ncol, n0, r, g, b, use, stats, k2, tempered, c_beg, hits, m, arg, s, w2, nan_seen); break;
            default: epi_block<1>(ea, tl, ch, ncol, n0, r, g, b, use, stats, k2, tempered, c_beg, hits, m, arg, s, w2, nan_seen); break;
          }
        }
      }
      // the accumulator may take the next tile's MMAs once every warp has read it
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(acc_empty + a);
      if (!stats) continue;
      // groups 1.. hand their statistics to group 0, which merges them in
      // column order (ties keep the lower column) and writes the tile's partial
      float* xb = xh + a * (kColGroups - 1) * 5 * BM;
      const int row = quad * 32 + lane;
      if (kColGroups > 1) {
        if (grp > 0) {
          float* x = xb + (grp - 1) * 5 * BM;
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
          const float mg = xb[(g - 1) * 5 * BM + row];
          if (mg > M) {
            M = mg;
            arg = __float_as_int(xb[(g - 1) * 5 * BM + 3 * BM + row]);
          }
          nan_seen |= xb[(g - 1) * 5 * BM + 4 * BM + row] != 0.f;
        }
        float S = 0.f, W2 = 0.f;
        if (tempered) {
          if (s > 0.f) {
            const float d = (m - M) * k2, sc = ex2_approx(d);
            S += sc * s;
            W2 += sc * fmaf(d, s, w2);
          }
          for (int g = 1; g < kColGroups; ++g) {
            const float* x = xb + (g - 1) * 5 * BM;
            const float mg = x[row], sg = x[BM + row], wg = x[2 * BM + row];
            if (sg > 0.f) {
              const float d = (mg - M) * k2, sc = ex2_approx(d);
              S += sc * sg;
              W2 += sc * fmaf(d, sg, wg);
            }
          }
        }
        if (sh.n_mt > 1) {
          if (nan_seen) S = __int_as_float(0x7fc00000);
          ea.part[static_cast<size_t>(r) * ea.n_nt + n_t] = make_float4(M, S, W2 * kLn2, __int_as_float(arg));
        } else {
          // one row tile: every tile of this CTA has the same rows, so the CTA
          // folds its tiles into one partial (ties keep the lower column)
          if (M > run_m || (M == run_m && arg < run_arg)) {
            if (tempered && run_s > 0.f) {
              const float d = (run_m - M) * k2, sc = ex2_approx(d);
              run_w2 = sc * fmaf(d, run_s, run_w2);
              run_s *= sc;
            }
            run_m = M;
            run_arg = arg;
          }
          if (tempered && S > 0.f) {
            const float d = (M - run_m) * k2, sc = ex2_approx(d);
            run_s += sc * S;
            run_w2 += sc * fmaf(d, S, W2);
          }
          run_nan |= nan_seen;
          if (t + static_cast<int>(gridDim.x) >= sh.n_tiles)
            ea.part[static_cast<size_t>(r) * ea.n_nt + blockIdx.x] =
                make_float4(run_m, run_nan ? __int_as_float(0x7fc00000) : run_s, run_w2 * kLn2, __int_as_float(run_arg));
        }
        if ((!ok || failed(&s_fail)) && ea.dev_status) atomicOr(ea.dev_status + b, MEDUSA_DEV_TIMEOUT);
      }
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
  const float4* part;  // [R, n_nt] statistics partials (n_nt of them per row)
  int n_nt, R;
  float4* rowst;       // [R] merged statistics
  unsigned char* acc;  // [R] typical-acceptance test of each node against its parent (root: 1)
  float* logp;         // [R] ln p of each node under its parent (root: 0)
  int joint;           // tie-break among the deepest kept nodes: 0 first in order, 1 highest joint probability
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
  // the KV commit of the accepted path, run by the same CTA (k_cache NULL: none)
  const uint4* k_new;
  const uint4* v_new;
  uint4* k_cache;
  uint4* v_cache;
  int32_t* kv_len;
  int Hkv, row_vecs, Lmax;
};

// ------------------------------------------------------------------------
// K6b: longest kept prefix of request b and the next root (whole CTA; every
// node's own acceptance test is in a.acc, the merged statistics in a.rowst).
// A node is kept when it and all its ancestors passed; the deepest kept node
// wins, ties to the lowest canonical index.
// ------------------------------------------------------------------------
__device__ inline uint32_t ordered_bits(float f) {  // monotone map of floats to unsigned (NaN lowest)
  if (f != f) return 0u;
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ void accept_request(const AcceptArgs& a, int b, unsigned char* s_acc, const int16_t* s_par,
                               const int16_t* s_dep, const int16_t* s_fp, float* s_lp, int* s_chain,
                               unsigned long long* s_best) {
  const medusa_tree_dev& tr = a.tr;
  const int T = tr.T;
  const size_t base = static_cast<size_t>(b) * T;
  if (threadIdx.x == 0) *s_best = 0ull;
  for (int c = threadIdx.x; c < T; c += blockDim.x) {
    s_acc[c] = __ldcg(a.acc + base + c);
    if (a.joint) s_lp[c] = c == 0 ? 0.f : __ldcg(a.logp + base + c);
  }
  __syncthreads();
  for (int d = 1; d <= tr.dmax; ++d) {
    for (int c = threadIdx.x; c < T; c += blockDim.x)
      if (s_dep[c] == d) {
        s_acc[c] = s_acc[c] && s_acc[s_par[c]];
        if (a.joint) s_lp[c] += s_lp[s_par[c]];  // ln of the path's joint probability
      }
    __syncthreads();
  }
  // key: depth, then (joint rule) the path's log probability, then the lowest index
  unsigned long long key = 0xFFFFull;  // root: depth 0, index 0
  for (int c = threadIdx.x; c < T; c += blockDim.x)
    if (s_acc[c]) {
      const unsigned long long lp = a.joint ? ordered_bits(s_lp[c]) : 0u;
      key = max(key, (static_cast<unsigned long long>(s_dep[c]) << 48) | (lp << 16) | (0xFFFFu - c));
    }
  for (int o = 16; o > 0; o >>= 1) key = max(key, __shfl_xor_sync(0xffffffffu, key, o));
  if ((threadIdx.x & 31) == 0) atomicMax(s_best, key);
  __syncthreads();
  const int best = 0xFFFF - static_cast<int>(*s_best & 0xFFFFull);
  const int a_len = s_dep[best];
  if (threadIdx.x == 0) {
    int node = best;
    for (int d = a_len; d >= 0; --d) {
      s_chain[d] = node;
      node = s_par[node];
    }
  }
  __syncthreads();
  // accepted tokens root..best, -1 past the winner
  int32_t* out = a.accepted_tokens + static_cast<size_t>(b) * (tr.dmax + 1);
  for (int d = threadIdx.x; d <= tr.dmax; d += blockDim.x) out[d] = d <= a_len ? a.tokens[base + s_chain[d]] : -1;
  if (threadIdx.x == 32) {  // a second warp, beside the token reads of the first
    a.next_root[b] = __float_as_int(__ldcg(a.rowst + base + best).w);
    a.accept_len[b] = a_len;
    a.best_node[b] = best;
    a.best_path[b] = s_fp[best];
  }
  if (a.k_cache) {
    // the commit (what medusa_kv_commit does): the path's K/V rows root..best go to
    // cache positions kv_len..kv_len+a_len, then kv_len advances; a request whose
    // rows would pass Lmax is flagged and its cache left untouched
    __shared__ int s_L;
    if (threadIdx.x == 0) {
      const int L = a.kv_len[b];
      s_L = (L < 0 || L + a_len + 1 > a.Lmax) ? -1 : L;
      if (s_L < 0 && a.dev_status) atomicOr(a.dev_status + b, MEDUSA_DEV_KV_OVERFLOW);
    }
    __syncthreads();
    const int L = s_L;
    if (L >= 0) {
      const int per_d = a.Hkv * a.row_vecs, total = (a_len + 1) * per_d;
      constexpr int U = 4;  // all loads of a round before its stores
      for (int e0 = threadIdx.x; e0 < total; e0 += blockDim.x * U) {
        uint4 kr[U], vr[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int e = e0 + u * blockDim.x;
          if (e < total) {
            const int d = e / per_d, g = (e / a.row_vecs) % a.Hkv, j = e % a.row_vecs;
            const size_t src = ((base + s_chain[d]) * a.Hkv + g) * a.row_vecs + j;
            kr[u] = a.k_new[src];
            vr[u] = a.v_new[src];
          }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int e = e0 + u * blockDim.x;
          if (e < total) {
            const int d = e / per_d, g = (e / a.row_vecs) % a.Hkv, j = e % a.row_vecs;
            const size_t dst = ((static_cast<size_t>(b) * a.Hkv + g) * a.Lmax + L + d) * a.row_vecs + j;
            a.k_cache[dst] = kr[u];
            a.v_cache[dst] = vr[u];
          }
        }
      }
      __syncthreads();
      if (threadIdx.x == 0) a.kv_len[b] = L + a_len + 1;
    }
  }
  __syncthreads();
}

// ------------------------------------------------------------------------
// K6: merge each node's tile statistics (warp per node, kMergeRows nodes per
// CTA), then test the node's children against them: at temperature > 0
// child c passes when p(c) = softmax(z/tau)[token c] exceeds
// min(threshold, alpha * exp(-H)) with H the entropy of the same
// distribution; at temperature 0 when its token is the argmax.  The last CTA
// to finish a request's nodes (ticket per request) then runs K6b for it.
// ------------------------------------------------------------------------
constexpr int kMergeRows = 8;

__global__ void __launch_bounds__(kMergeRows * 32) merge_accept_kernel(AcceptArgs a) {
  // shared: parent[T], depth[T], first path[T] (int16; the tree tables are constant,
  // so they are read before the wait on the preceding kernel), then kept[T] bytes
  extern __shared__ __align__(16) unsigned char accept_smem[];
  const int T = a.tr.T;
  int16_t* s_par = reinterpret_cast<int16_t*>(accept_smem);
  int16_t* s_dep = s_par + T;
  int16_t* s_fp = s_dep + T;
  float* s_lp = reinterpret_cast<float*>(s_fp + T + (T & 1));  // 4-byte aligned after three int16 arrays
  unsigned char* s_acc = reinterpret_cast<unsigned char*>(s_lp + T);
  __shared__ int s_chain[MEDUSA_MAX_DEPTH + 1];
  __shared__ unsigned long long s_best;
  __shared__ int s_last;
  for (int c = threadIdx.x; c < T; c += blockDim.x) {
    s_par[c] = static_cast<int16_t>(a.tr.parent[c]);
    s_dep[c] = static_cast<int16_t>(a.tr.depth[c]);
    s_fp[c] = static_cast<int16_t>(a.tr.first_path[c]);
  }
  const int r0 = blockIdx.x * kMergeRows, r1 = min(a.R, r0 + kMergeRows);
  const int r = r0 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  int c_beg = 0, c_cnt = 0;
  if (r < r1) {
    const int node = r % T;
    c_beg = a.tr.child_start[node];
    c_cnt = a.tr.child_count[node];
  }
  pdl_wait();
  pdl_trigger();
  if (r < r1) {
    const int b = r / T, node = r % T;
    const size_t base = static_cast<size_t>(b) * T;
    // the first 32 children's tokens and logits load beside the partials
    int tok = 0;
    float cz = 0.f;
    if (lane < c_cnt) {
      tok = a.tokens[base + c_beg + lane];
      cz = a.child_z[base + c_beg + lane];
    }
    const float4 v = merge_row(a.part + static_cast<size_t>(r) * a.n_nt, a.n_nt, a.inv_tau);
    const bool tempered = a.inv_tau > 0.f;
    const float H = tempered ? logf(v.y) - v.z / v.y : 0.f;
    const float thr = fminf(a.thr, a.alpha * expf(-H));
    if (lane == 0) {
      a.rowst[r] = v;
      if (a.node_H) a.node_H[base + node] = H;
      if (node == 0) {
        a.acc[base] = 1;
        if (a.node_p) a.node_p[base] = 1.f;
      }
      if ((v.x != v.x || v.y != v.y) && a.dev_status) atomicOr(a.dev_status + b, MEDUSA_DEV_NAN);
    }
    for (int k = lane; k < c_cnt; k += 32) {
      if (k >= 32) {
        tok = a.tokens[base + c_beg + k];
        cz = a.child_z[base + c_beg + k];
      }
      bool pass;
      float p;
      if (tempered) {
        p = expf((cz - v.x) * a.inv_tau) / v.y;
        pass = p > thr;
      } else {
        pass = tok == __float_as_int(v.w);
        p = pass ? 1.f : 0.f;
      }
      a.acc[base + c_beg + k] = pass ? 1 : 0;
      if (a.joint) a.logp[base + c_beg + k] = logf(p);
      if (a.node_p) a.node_p[base + c_beg + k] = p;
    }
  }
  __threadfence();
  __syncthreads();
  for (int b = r0 / T; b <= (r1 - 1) / T; ++b) {
    const int need = ((b + 1) * T - 1) / kMergeRows - (b * T) / kMergeRows + 1;  // CTAs holding b's nodes
    if (threadIdx.x == 0) s_last = atomicAdd(a.tickets + b, 1) == need - 1;
    __syncthreads();
    if (s_last) {
      __threadfence();
      accept_request(a, b, s_acc, s_par, s_dep, s_fp, s_lp, s_chain, &s_best);
      if (threadIdx.x == 0) a.tickets[b] = 0;  // ready for the next launch
    }
    __syncthreads();
  }
}

constexpr size_t kTcSmemMax = 227 * 1024 - 1024;  // the kernel's static shared memory takes 1 KB
constexpr size_t kTcFixedBytes = 1024 + (2 * kMaxStagesW + 2 * kMaxStagesX + 4) * 8 + 16 + kXchgBytes;

TcShape tc_shape(const VerifyPlan& p, bool topk = false) {
  TcShape sh{};
  sh.topk = topk ? 1 : 0;
  sh.BN = p.BN;
  sh.qr = p.qr;
  sh.n_mt = p.n_mt;
  sh.n_nt = p.n_nt;
  sh.n_g = p.n_g;
  sh.n_tiles = p.n_tiles;
  const size_t wb = static_cast<size_t>(p.BN) * BK * 2;
  // three X stages (L2 latency); the rest of shared memory goes to the weight
  // ring, which also carries the prefetch made before the dependency wait
  sh.sx = 3;
  const size_t fixed = kTcFixedBytes + (topk ? kTopkBufBytes : 0);
  sh.sw = static_cast<int>(std::min<size_t>(kMaxStagesW, (kTcSmemMax - fixed - sh.sx * kXStageBytes) / wb));
  return sh;
}

size_t tc_smem_bytes(const TcShape& sh) {
  return kTcFixedBytes + (sh.topk ? kTopkBufBytes : 0) + static_cast<size_t>(sh.sx) * kXStageBytes +
         static_cast<size_t>(sh.sw) * sh.BN * BK * 2;
}

template <int BN, bool TOPK>
int launch_tc(const VerifyPlan& p, const CUtensorMap& mx, const CUtensorMap& mw, int H, const EpiArgs& ea,
              cudaStream_t st) {
  const TcShape sh = tc_shape(p, TOPK);
  if (sh.sw < 2) return MEDUSA_ERR_UNSUPPORTED;
  const size_t smem = tc_smem_bytes(sh);
  auto k = verify_tc_kernel<BN, TOPK>;
  if (!ensure_dyn_smem(k, smem))
    return MEDUSA_ERR_CUDA;
  if (launch_pdl(k, dim3(p.grid), dim3(kTcThreads), smem, st, mx, mw, H, sh, ea) != cudaSuccess) {
    (void)cudaGetLastError();
    return MEDUSA_ERR_CUDA;
  }
  MEDUSA_LAUNCH_CHECK();
  return MEDUSA_OK;
}

int dispatch_tc(const VerifyPlan& p, const CUtensorMap& mx, const CUtensorMap& mw, int H, const EpiArgs& ea,
                cudaStream_t st) {
  if (ea.topk_k > 0) {
    if (ea.topk_k > kEpiTopkMax || !ea.cand_v || !ea.cand_i) return MEDUSA_ERR_INVALID_ARG;
    switch (p.BN) {
#define MEDUSA_BN(n) case n: return launch_tc<n, true>(p, mx, mw, H, ea, st);
      MEDUSA_BN(128) MEDUSA_BN(160) MEDUSA_BN(192) MEDUSA_BN(224) MEDUSA_BN(256)
#undef MEDUSA_BN
      default: return MEDUSA_ERR_UNSUPPORTED;
    }
  }
  switch (p.BN) {
#define MEDUSA_BN(n) case n: return launch_tc<n, false>(p, mx, mw, H, ea, st);
    MEDUSA_BN(16) MEDUSA_BN(32) MEDUSA_BN(48) MEDUSA_BN(64) MEDUSA_BN(80) MEDUSA_BN(96) MEDUSA_BN(112)
    MEDUSA_BN(128) MEDUSA_BN(144) MEDUSA_BN(160) MEDUSA_BN(176) MEDUSA_BN(192) MEDUSA_BN(208) MEDUSA_BN(224)
    MEDUSA_BN(240) MEDUSA_BN(256)
#undef MEDUSA_BN
    default: return MEDUSA_ERR_UNSUPPORTED;
  }
}

// ------------------------------------------------------------------------
// Nucleus (top-p) draw of the next token from the accepted node's logits, with
// the uniform draw given: one CTA per request.  The nucleus is the shortest run
// of tokens in descending probability (equal values by the lower id) whose mass
// reaches top_p; the draw picks by inverse CDF over the renormalised nucleus,
// tokens in ascending id order.  The nucleus edge is found by bisection on the
// ordered bit patterns of the logits (mass(z >= t) is monotone in t), tied
// tokens at the edge are taken by id, and the draw uses a block scan.
// ------------------------------------------------------------------------
constexpr int kSampleThreads = 1024;

__device__ inline uint32_t to_ordered(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ inline float from_ordered(uint32_t o) {
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7fffffffu) : ~o);
}

// Block-wide sum (all threads receive it).
__device__ inline float block_sum(float v, float* red) {
  v = warp_sum(v);
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[w] = v;
  __syncthreads();
  float t = lane < static_cast<int>(blockDim.x >> 5) ? red[lane] : 0.f;
  return warp_sum(t);
}

// Block-wide exclusive prefix sum of one value per thread (and the total).
template <typename U>
__device__ inline U block_excl_scan(U v, U* red, U& total) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  U x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const U y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  __syncthreads();
  if (lane == 31) red[w] = x;
  __syncthreads();
  if (w == 0) {
    U t = lane < static_cast<int>(blockDim.x >> 5) ? red[lane] : U(0);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const U y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    red[lane] = t;  // inclusive prefix of warp sums
  }
  __syncthreads();
  total = red[(blockDim.x >> 5) - 1];
  return (w > 0 ? red[w - 1] : U(0)) + x - v;
}

__global__ void __launch_bounds__(kSampleThreads) nucleus_next_kernel(const float* __restrict__ logits,
                                                                      const int32_t* __restrict__ best,
                                                                      const float* __restrict__ uniform, int T, int V,
                                                                      float inv_tau, float top_p,
                                                                      int32_t* __restrict__ next_token) {
  __shared__ float s_redf[32];
  __shared__ int s_redi[32];
  __shared__ float s_m;
  __shared__ int s_arg;
  const int b = blockIdx.x;
  pdl_wait();
  pdl_trigger();
  const int node = min(max(best[b], 0), T - 1);
  const float* z = logits + (static_cast<size_t>(b) * T + node) * V;
  // maximum (first on ties) and minimum
  float m = -INFINITY, mn = INFINITY;
  int arg = 0x7fffffff;
  for (int v = threadIdx.x; v < V; v += blockDim.x) {
    const float x = z[v];
    if (better(x, v, m, arg)) { m = x; arg = v; }
    mn = fminf(mn, x);
  }
  warp_argmax(m, arg);
  for (int o = 16; o > 0; o >>= 1) mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __shared__ float s_min[32];
  if (lane == 0) { s_redf[w] = m; s_redi[w] = arg; s_min[w] = mn; }
  __syncthreads();
  if (threadIdx.x == 0) {
    float bm = -INFINITY;
    int ba = 0x7fffffff;
    for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i)
      if (better(s_redf[i], s_redi[i], bm, ba)) { bm = s_redf[i]; ba = s_redi[i]; }
    s_m = bm;
    s_arg = ba;
  }
  __syncthreads();
  const float M = s_m;
  if (inv_tau == 0.f) {
    if (threadIdx.x == 0) next_token[b] = s_arg;
    return;
  }
  float zmin = s_min[0];
  for (int i = 1; i < static_cast<int>(blockDim.x >> 5); ++i) zmin = fminf(zmin, s_min[i]);
  const float k2 = inv_tau * 1.4426950408889634f;
  auto q_of = [&](float x) { return ex2_approx((x - M) * k2); };
  // mass of the tokens whose logit is at least t (unnormalised)
  auto mass_ge = [&](float t) {
    float acc = 0.f;
    for (int v = threadIdx.x; v < V; v += blockDim.x) {
      const float x = z[v];
      acc += x >= t ? q_of(x) : 0.f;
    }
    return block_sum(acc, s_redf);
  };
  const float S = mass_ge(-INFINITY);
  const float goal = top_p * S;
  // largest t (a logit value) with mass(z >= t) >= goal: the smallest logit of the nucleus
  uint32_t lo = to_ordered(zmin), hi = to_ordered(M);
  if (top_p < 1.f) {
    while (lo < hi) {
      const uint32_t mid = lo + (hi - lo + 1) / 2;
      if (mass_ge(from_ordered(mid)) >= goal) lo = mid; else hi = mid - 1;
    }
  }
  const float tstar = from_ordered(lo);
  // tokens tied at the edge join by id until the mass is reached
  float above = 0.f;
  int ties = 0;
  for (int v = threadIdx.x; v < V; v += blockDim.x) {
    const float x = z[v];
    above += x > tstar ? q_of(x) : 0.f;
    ties += x == tstar;
  }
  above = block_sum(above, s_redf);
  int n_ties = 0;
  {
    int tt = ties;
    for (int o = 16; o > 0; o >>= 1) tt += __shfl_xor_sync(0xffffffffu, tt, o);
    __syncthreads();
    if (lane == 0) s_redi[w] = tt;
    __syncthreads();
    for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i) n_ties += s_redi[i];
  }
  const float qt = q_of(tstar);
  int take = top_p >= 1.f ? n_ties : static_cast<int>(ceilf((goal - above) / qt));
  take = min(max(take, 1), n_ties);
  const float nmass = above + take * qt;
  const float target = uniform[b] * nmass;
  // inverse CDF in id order: each thread a contiguous chunk of ids
  const int C = cdiv(V, blockDim.x);
  const int v0 = min(V, static_cast<int>(threadIdx.x) * C), v1 = min(V, v0 + C);
  int my_ties = 0;
  for (int v = v0; v < v1; ++v) my_ties += z[v] == tstar;
  __syncthreads();
  int ties_total = 0;
  const int tie_before = block_excl_scan<int>(my_ties, s_redi, ties_total);
  float my_mass = 0.f;
  {
    int tr = tie_before;
    for (int v = v0; v < v1; ++v) {
      const float x = z[v];
      const bool in = x > tstar || (x == tstar && tr++ < take);
      my_mass += in ? q_of(x) : 0.f;
    }
  }
  __syncthreads();
  float mass_total = 0.f;
  const float before = block_excl_scan<float>(my_mass, s_redf, mass_total);
  const bool last_chunk = v1 >= V || (threadIdx.x + 1) * C >= V;
  if ((before <= target && target < before + my_mass) || (last_chunk && target >= before + my_mass && v0 < V)) {
    // the draw falls in this chunk (or past the total by rounding: the last member)
    float run = before;
    int tr = tie_before, pick = -1, last_member = -1;
    for (int v = v0; v < v1; ++v) {
      const float x = z[v];
      const bool in = x > tstar || (x == tstar && tr++ < take);
      if (!in) continue;
      last_member = v;
      run += q_of(x);
      if (run > target) { pick = v; break; }
    }
    if (pick < 0) pick = last_member;
    if (pick >= 0) next_token[b] = pick;
  }
}

}  // namespace

MEDUSA_API int medusa_sample_next(const medusa_tree* tree, const float* logits, const int32_t* best_node,
                                  const float* uniform, int32_t B, int32_t V, float temperature, float top_p,
                                  int32_t* next_token, medusa_stream_t stream) {
  if (!tree || !logits || !best_node || !uniform || !next_token) return MEDUSA_ERR_INVALID_ARG;
  if (B < 1 || B > MEDUSA_MAX_BATCH || V < 1 || !(temperature >= 0.f) || !(top_p > 0.f && top_p <= 1.f))
    return MEDUSA_ERR_INVALID_ARG;
  const void* ptrs[] = {logits, best_node, uniform, next_token};
  for (const void* q : ptrs)
    if (!aligned16(q)) return MEDUSA_ERR_ALIGNMENT;
  const float inv_tau = temperature > 0.f ? 1.f / temperature : 0.f;
  if (launch_pdl(nucleus_next_kernel, dim3(B), dim3(kSampleThreads), 0, reinterpret_cast<cudaStream_t>(stream), logits,
                 best_node, uniform, tree->T, V, inv_tau, top_p, next_token) != cudaSuccess) {
    (void)cudaGetLastError();
    return MEDUSA_ERR_CUDA;
  }
  MEDUSA_LAUNCH_CHECK();
  return MEDUSA_OK;
}

namespace medusa {

int launch_group_logits_bf16(const void* x, int R, int n_g, const void* w, int H, int V, float* logits,
                             cudaStream_t st) {
  if (!x || !w || !logits || R < 1 || n_g < 1 || V < 1 || H < 8 || H % 8 != 0)
    return MEDUSA_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w) || !aligned16(logits)) return MEDUSA_ERR_ALIGNMENT;
  const VerifyPlan p = plan_tc(R, n_g, V);
  CUtensorMap mx, mw;
  const bool okx = n_g == 1 ? make_tmap_bf16(&mx, x, R, H, p.qr)
                            : make_tmap_bf16_3d(&mx, x, H, n_g, R, static_cast<uint64_t>(H) * 2,
                                                static_cast<uint64_t>(n_g) * H * 2, 1, p.qr);
  if (!okx || !make_tmap_bf16(&mw, w, static_cast<uint64_t>(n_g) * V, H, p.BN)) return MEDUSA_ERR_CUDA;
  const EpiArgs ea{R, V, 1, 0, nullptr, medusa_tree_dev{}, 0.f, logits, nullptr, nullptr, nullptr, n_g};
  return dispatch_tc(p, mx, mw, H, ea, st);
}

int group_topk_tiles(int R, int n_g, int V) { return plan_tc(R, n_g, V, true).n_nt; }

int launch_group_topk_bf16(const void* x, int R, int n_g, const void* w, int H, int V, int k, float* cand_v,
                           int* cand_i, float* logits, cudaStream_t st) {
  if (!x || !w || !cand_v || !cand_i || R < 1 || n_g < 1 || V < 1 || H < 8 || H % 8 != 0 || k < 1 ||
      k > kEpiTopkMax)
    return MEDUSA_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w) || (logits && !aligned16(logits))) return MEDUSA_ERR_ALIGNMENT;
  const VerifyPlan p = plan_tc(R, n_g, V, true);
  CUtensorMap mx, mw;
  const bool okx = n_g == 1 ? make_tmap_bf16(&mx, x, R, H, p.qr)
                            : make_tmap_bf16_3d(&mx, x, H, n_g, R, static_cast<uint64_t>(H) * 2,
                                                static_cast<uint64_t>(n_g) * H * 2, 1, p.qr);
  if (!okx || !make_tmap_bf16(&mw, w, static_cast<uint64_t>(n_g) * V, H, p.BN)) return MEDUSA_ERR_CUDA;
  const EpiArgs ea{R, V, 1, p.n_nt, nullptr, medusa_tree_dev{}, 0.f, logits, nullptr, nullptr, nullptr, n_g, k,
                   cand_v, cand_i};
  return dispatch_tc(p, mx, mw, H, ea, st);
}

}  // namespace medusa

MEDUSA_API size_t medusa_verify_accept_workspace_size(const medusa_tree* tree, int32_t B, int32_t H, int32_t V,
                                                      medusa_dtype dtype) {
  if (!tree || B < 1 || H < 1 || V < 1) return 0;
  VerifyPlan p = plan_verify(B, tree->T, V, dtype);
  return carve_verify_ws(nullptr, p, V, dtype).bytes;
}

namespace {

struct CommitArgs {
  const void* k_new;
  const void* v_new;
  void* k_cache;
  void* v_cache;
  int32_t* kv_len;
  int Hkv, D, Lmax;
};

int verify_accept_impl(const medusa_tree* tree, const void* x, const void* lm_head, const int32_t* tree_tokens,
                       int32_t B, int32_t H, int32_t V, medusa_dtype dtype, float temperature,
                       float posterior_threshold, float posterior_alpha, int32_t tie_break, float* logits,
                       float* node_p, float* node_H, int32_t* accept_len, int32_t* best_path, int32_t* best_node,
                       int32_t* accepted_tokens, int32_t* next_root, int32_t* dev_status, void* ws, size_t ws_bytes,
                       medusa_stream_t stream, const CommitArgs* cm) {
  if (!tree || !x || !lm_head || !tree_tokens || !accept_len || !best_path || !best_node || !accepted_tokens ||
      !next_root)
    return MEDUSA_ERR_INVALID_ARG;
  if (B < 1 || B > MEDUSA_MAX_BATCH || H < 8 || V < 1 || !(temperature >= 0.f)) return MEDUSA_ERR_INVALID_ARG;
  if (tie_break != 0 && tie_break != 1) return MEDUSA_ERR_INVALID_ARG;
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
  EpiArgs ea{p.R, V, T, p.n_parts, tree_tokens, tree->dev, inv_tau, logits, w.part, w.child_z, dev_status, 1};

  if (dtype == MEDUSA_BF16) {
    CUtensorMap mx, mw;
    if (!make_tmap_bf16(&mx, x, p.R, H, p.qr) || !make_tmap_bf16(&mw, lm_head, V, H, p.BN))
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
  AcceptArgs aa{tree->dev, tree_tokens, w.part, p.n_parts, p.R, w.rowst, w.acc, w.logp, tie_break, w.tickets,
                w.child_z, inv_tau, posterior_threshold, posterior_alpha, node_p, node_H, accept_len, best_path,
                best_node, accepted_tokens, next_root, dev_status};
  if (cm) {
    const int es = dtype == MEDUSA_BF16 ? 2 : 4;
    aa.k_new = static_cast<const uint4*>(cm->k_new);
    aa.v_new = static_cast<const uint4*>(cm->v_new);
    aa.k_cache = static_cast<uint4*>(cm->k_cache);
    aa.v_cache = static_cast<uint4*>(cm->v_cache);
    aa.kv_len = cm->kv_len;
    aa.Hkv = cm->Hkv;
    aa.row_vecs = cm->D * es / 16;
    aa.Lmax = cm->Lmax;
  }
  const size_t accept_smem = static_cast<size_t>(T) * 6 + (T & 1) * 2 + static_cast<size_t>(T) * 5;
  if (launch_pdl(merge_accept_kernel, dim3(cdiv(p.R, kMergeRows)), dim3(kMergeRows * 32), accept_smem, st, aa) !=
      cudaSuccess) {
    (void)cudaGetLastError();
    return MEDUSA_ERR_CUDA;
  }
  MEDUSA_LAUNCH_CHECK();
  return MEDUSA_OK;
}

}  // namespace

MEDUSA_API int medusa_verify_accept(const medusa_tree* tree, const void* x, const void* lm_head,
                                    const int32_t* tree_tokens, int32_t B, int32_t H, int32_t V, medusa_dtype dtype,
                                    float temperature, float posterior_threshold, float posterior_alpha,
                                    int32_t tie_break, float* logits, float* node_p, float* node_H, int32_t* accept_len,
                                    int32_t* best_path, int32_t* best_node, int32_t* accepted_tokens,
                                    int32_t* next_root, int32_t* dev_status, void* ws, size_t ws_bytes,
                                    medusa_stream_t stream) {
  return verify_accept_impl(tree, x, lm_head, tree_tokens, B, H, V, dtype, temperature, posterior_threshold,
                            posterior_alpha, tie_break, logits, node_p, node_H, accept_len, best_path, best_node,
                            accepted_tokens, next_root, dev_status, ws, ws_bytes, stream, nullptr);
}

MEDUSA_API int medusa_verify_accept_commit(const medusa_tree* tree, const void* x, const void* lm_head,
                                           const int32_t* tree_tokens, int32_t B, int32_t H, int32_t V,
                                           medusa_dtype dtype, float temperature, float posterior_threshold,
                                           float posterior_alpha, int32_t tie_break, float* logits, float* node_p,
                                           float* node_H, int32_t* accept_len, int32_t* best_path,
                                           int32_t* best_node, int32_t* accepted_tokens, int32_t* next_root,
                                           int32_t* dev_status, const void* k_new, const void* v_new, void* k_cache,
                                           void* v_cache, int32_t* kv_len, int32_t Hkv, int32_t D, int32_t Lmax,
                                           void* ws, size_t ws_bytes, medusa_stream_t stream) {
  if (!k_new || !v_new || !k_cache || !v_cache || !kv_len) return MEDUSA_ERR_INVALID_ARG;
  if (Hkv < 1 || D < 1 || Lmax < 0) return MEDUSA_ERR_INVALID_ARG;
  const int es = dtype == MEDUSA_BF16 ? 2 : 4;
  if ((D * es) % 16 != 0) return MEDUSA_ERR_UNSUPPORTED;
  const void* ptrs[] = {k_new, v_new, k_cache, v_cache, kv_len};
  for (const void* q : ptrs)
    if (!aligned16(q)) return MEDUSA_ERR_ALIGNMENT;
  const CommitArgs cm{k_new, v_new, k_cache, v_cache, kv_len, Hkv, D, Lmax};
  return verify_accept_impl(tree, x, lm_head, tree_tokens, B, H, V, dtype, temperature, posterior_threshold,
                            posterior_alpha, tie_break, logits, node_p, node_H, accept_len, best_path, best_node,
                            accepted_tokens, next_root, dev_status, ws, ws_bytes, stream, &cm);
}
