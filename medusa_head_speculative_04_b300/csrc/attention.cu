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
// bf16 path: one persistent-style launch over a balanced split of all key
// tiles.  The work of a request's KV head is a sequence of 64-key tiles: the
// kv_len cached keys, then the tree's own keys (masked by the cached ancestor
// bitmask; tiles no query row of the tile can see are skipped).  Every CTA
// takes an equal share of the concatenated tile sequence of all requests and
// heads, computed on the device from kv_len, so ragged batches stay balanced.
// A query tile holds up to 128 rows (node, query head of the KV head's group):
// heads that share a KV head share every K/V tile.  One producer warp streams
// K/V tiles into shared memory with TMA (128-byte swizzled boxes, mbarrier
// completion, kStages deep); each consumer warp owns 16 query rows and runs
// QK^T and PV on mma.sync bf16 tiles with an fp32 online softmax.  A head
// whose tiles all fall to one CTA is written out directly; a head split over
// several CTAs leaves one partial (unnormalised output, running max and sum)
// per CTA, and a combine launch merges them (one warp per output row, every
// partial's loads in flight at once).
// fp32 path: an exact scalar kernel (small shapes).
#include <algorithm>
#include <cmath>

#include "tc.cuh"
#include "tree.cuh"

using namespace medusa;

namespace {

constexpr int KB = 64;          // keys per tile
constexpr int kStages = 3;      // K/V tiles in flight per CTA
constexpr int kCtasPerSm = 2;
constexpr int kMaxWarps = 8;    // consumer warps: 128 query rows
constexpr int kMaxSplit = 320;  // CTAs of a split (2 per SM, up to 160 SMs)

struct AttnPlan {
  int G, R, n_qt, rpt, W, ntt, nctas, units;
};

AttnPlan plan_attn(int T, int B, int Hq, int Hkv, int Lmax, int hint, int sms) {
  AttnPlan p{};
  p.G = Hq / Hkv;
  p.R = T * p.G;
  p.n_qt = cdiv(p.R, 16 * kMaxWarps);
  // rows per query tile: a multiple of 16 (mma.sync row blocks) and, when the
  // group divides 128, of the group size (a tile then starts at a node)
  const int gran = (128 % p.G == 0) ? std::max(16, p.G) : 16;
  p.rpt = cdiv(cdiv(p.R, p.n_qt), gran) * gran;
  p.W = p.rpt / 16;
  p.ntt = cdiv(T, KB);
  p.units = B * Hkv * p.n_qt;
  const int L = hint > 0 ? std::min(hint, Lmax) : Lmax;
  const long total = static_cast<long>(p.units) * (cdiv(std::max(L, 0), KB) + p.ntt);
  long n = std::min(std::min(static_cast<long>(kCtasPerSm) * sms, total), static_cast<long>(kMaxSplit));
  // A CTA whose range crosses from one unit into the next pays a second Q load
  // and O drain.  When every request has the same length, a grid that is a
  // multiple of the unit count puts every split point on a unit boundary.
  if (p.units <= n && n % p.units != 0) n = n / p.units * p.units;
  p.nctas = static_cast<int>(std::max(1L, n));
  return p;
}

// Partial results: a CTA's range starts and ends inside at most two split
// heads, so each CTA owns two slots: slot 0 for the head its range starts in,
// slot 1 for the head it ends in.
struct AttnWs {
  float* o_part;    // [nctas * 2 slots][rpt][D]
  float2* ml_part;  // [nctas * 2 slots][rpt] (running max, sum)
  size_t bytes;
};

AttnWs carve_attn_ws(void* base, const AttnPlan& p, int D) {
  AttnWs w{};
  size_t o = 0;
  auto take = [&](size_t n) { size_t s = o; o = align_up(o + n, 256); return s; };
  const size_t slots = static_cast<size_t>(p.nctas) * 2 * p.rpt;
  const size_t oo = take(slots * D * 4), om = take(slots * 8);
  char* c = static_cast<char*>(base);
  if (c) {
    w.o_part = reinterpret_cast<float*>(c + oo);
    w.ml_part = reinterpret_cast<float2*>(c + om);
  }
  w.bytes = o;
  return w;
}

constexpr int kMaxVisTiles = 128;  // query tiles whose tree visibility travels in the launch arguments

struct AttnArgs {
  medusa_tree_dev tr;
  int vis_known;                     // vis[] holds every query tile's visibility
  uint64_t vis[kMaxVisTiles];
  const __nv_bfloat16* q;
  const int32_t* kv_len;
  float* out;
  AttnWs ws;
  int32_t* dev_status;
  int B, T, Hq, Hkv, Lmax;
  float scale_log2;
  AttnPlan p;
};

__device__ inline uint32_t ld_u32(const __nv_bfloat16* p) { return *reinterpret_cast<const uint32_t*>(p); }

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

// A K or V tile in shared memory is D/64 TMA boxes of [64 keys][64 elements],
// each 8 KB, written with the 128-byte swizzle: 16-byte chunk c of key row j
// of a box sits at chunk position c ^ (j & 7).  `chunk` counts 16-byte chunks
// across the whole D-element row.
__device__ inline uint32_t tile_addr(uint32_t base, int key, int chunk) {
  return base + ((chunk >> 3) << 13) + key * 128 + (((chunk & 7) ^ (key & 7)) << 4);
}

// The split of the concatenated tile sequence: CTA c takes [start[c], start[c+1])
// with start[c] = c * total / n.  Built once per CTA in shared memory (the 64-bit
// divisions run in parallel), then the CTA holding position x is found by a
// binary search instead of a division.
__device__ inline void build_split(long long* s_start, long long total, int n) {
  for (int c = threadIdx.x; c <= n; c += blockDim.x) s_start[c] = static_cast<long long>(c) * total / n;
}
__device__ inline int split_cta_of(const long long* s_start, int n, long long x) {
  int lo = 0, hi = n - 1;  // largest c with start[c] <= x
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_start[mid] <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// One (request, KV head, query tile) unit met by a CTA: tiles [t0, t1) of its
// virtual tile sequence (nc cache tiles, then the tree tiles).
struct Seg {
  int b, g, qt, nc, t0, t1;
  long long ustart, uend;
};

__device__ inline bool next_seg(long long x, long long end, int& b, const AttnArgs& a, const int* s_len,
                                const long long* s_cum, Seg& s) {
  if (x >= end) return false;
  while (s_cum[b + 1] <= x) ++b;
  const int nc = cdiv(s_len[b], KB);
  const int cost = nc + a.p.ntt;
  const long long off = x - s_cum[b];
  const int ui = static_cast<int>(off / cost);
  s.b = b;
  s.g = ui / a.p.n_qt;
  s.qt = ui % a.p.n_qt;
  s.nc = nc;
  s.ustart = s_cum[b] + static_cast<long long>(ui) * cost;
  s.uend = s.ustart + cost;
  s.t0 = static_cast<int>(x - s.ustart);
  s.t1 = static_cast<int>((s.uend < end ? s.uend : end) - s.ustart);
  return true;
}

// Bit j set iff some query row of query tile qt may see a key of tree tile j
// (OR of the ancestor-mask rows of the tile's nodes).  Precomputed on the
// host for up to kMaxVisTiles query tiles, else computed here.  Whole warp.
__device__ inline uint64_t tree_tiles_visible(const AttnArgs& a, int qt) {
  if (a.vis_known) return a.vis[qt];
  const int lane = threadIdx.x & 31;
  const int r0 = qt * a.p.rpt, r1 = min(a.p.R, r0 + a.p.rpt);
  const int n0 = r0 / a.p.G, n1 = (r1 - 1) / a.p.G;
  const int mw = a.tr.mask_words;
  uint64_t bits = 0;
  for (int e = lane; e < (n1 - n0 + 1) * mw; e += 32) {
    const int node = n0 + e / mw, w = e % mw;
    if (a.tr.mask[static_cast<size_t>(node) * mw + w]) bits |= 1ull << (w >> 1);
  }
  const uint32_t lo = __reduce_or_sync(0xffffffffu, static_cast<uint32_t>(bits));
  const uint32_t hi = __reduce_or_sync(0xffffffffu, static_cast<uint32_t>(bits >> 32));
  return (static_cast<uint64_t>(hi) << 32) | lo;
}

template <int D>
__global__ void __launch_bounds__((kMaxWarps + 1) * 32, 1) tree_attn_kernel(
    const __grid_constant__ CUtensorMap tm_kc, const __grid_constant__ CUtensorMap tm_vc,
    const __grid_constant__ CUtensorMap tm_kt, const __grid_constant__ CUtensorMap tm_vt, AttnArgs a) {
  constexpr int NSUB = D / 64;
  constexpr uint32_t BOX = 64 * 128;
  constexpr uint32_t HALF = NSUB * BOX;  // one K (or V) tile
  constexpr uint32_t STAGE = 2 * HALF;
  extern __shared__ __align__(1024) unsigned char attn_smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(attn_smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * STAGE);
  uint64_t* empty = full + kStages;
  __shared__ int s_len[MEDUSA_MAX_BATCH];
  __shared__ long long s_cum[MEDUSA_MAX_BATCH + 1];
  __shared__ long long s_start[kMaxSplit + 1];

  const AttnPlan& p = a.p;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int W = p.W;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(full + s, 1);
      tc::mbar_init(empty + s, W);
    }
    tc::fence_mbar_init();
    tc::prefetch_tmap(&tm_kc);
    tc::prefetch_tmap(&tm_vc);
    tc::prefetch_tmap(&tm_kt);
    tc::prefetch_tmap(&tm_vt);
  }
  pdl_wait();
  for (int b = threadIdx.x; b < a.B; b += blockDim.x) s_len[b] = min(max(a.kv_len[b], 0), a.Lmax);
  __syncthreads();
  if (threadIdx.x == 0) {
    long long c = 0;
    const int upb = a.Hkv * p.n_qt;
    for (int b = 0; b < a.B; ++b) {
      s_cum[b] = c;
      c += static_cast<long long>(upb) * (cdiv(s_len[b], KB) + p.ntt);
    }
    s_cum[a.B] = c;
  }
  __syncthreads();
  pdl_trigger();
  const long long total = s_cum[a.B];
  // the grid was sized from an upper bound of kv_len: with fewer tiles than
  // CTAs only the first `total` CTAs take part, so that every range is non-empty
  const int nct = static_cast<int>(min(static_cast<long long>(gridDim.x), total));
  build_split(s_start, total, nct);
  __syncthreads();
  if (static_cast<int>(blockIdx.x) >= nct) return;
  const long long start = s_start[blockIdx.x], end = s_start[blockIdx.x + 1];

  if (warp == W) {
    // ---------------- producer: TMA loads of K/V tiles ----------------
    int stage = 0, issued = 0;
    uint32_t phase = 0;
    bool fail = false;
    int b = 0;
    Seg sg;
    for (long long x = start; !fail && next_seg(x, end, b, a, s_len, s_cum, sg); x = sg.ustart + sg.t1) {
      const uint64_t vis = tree_tiles_visible(a, sg.qt);
      if (lane == 0) {
        for (int t = sg.t0; t < sg.t1; ++t) {
          const bool tree = t >= sg.nc;
          const int j = t - sg.nc;
          if (tree && !((vis >> j) & 1ull)) continue;
          if (!tc::mbar_wait(empty + stage, phase ^ 1)) { fail = true; break; }
          tc::mbar_expect_tx(full + stage, STAGE);
          const uint32_t sk = smem_u32(smem + stage * STAGE), sv = sk + HALF;
#pragma unroll
          for (int h = 0; h < NSUB; ++h) {
            if (!tree) {
              const int z = sg.b * a.Hkv + sg.g;
              tc::tma_load_3d(sk + h * BOX, &tm_kc, 64 * h, t * KB, z, full + stage);
              tc::tma_load_3d(sv + h * BOX, &tm_vc, 64 * h, t * KB, z, full + stage);
            } else {
              const int z = sg.b * a.T + j * KB;
              tc::tma_load_3d(sk + h * BOX, &tm_kt, 64 * h, sg.g, z, full + stage);
              tc::tma_load_3d(sv + h * BOX, &tm_vt, 64 * h, sg.g, z, full + stage);
            }
          }
          ++issued;
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
      }
      fail = __shfl_sync(0xffffffffu, fail, 0);
    }
    if (lane == 0) {
      // every issued copy must have landed before the CTA's shared memory goes away
      for (int i = 0; i < min(issued, kStages); ++i) {
        const int k = issued - 1 - i;
        if (!tc::mbar_wait(full + (k % kStages), static_cast<uint32_t>((k / kStages) & 1))) fail = true;
      }
      if (fail && a.dev_status) atomicOr(a.dev_status, MEDUSA_DEV_TIMEOUT);
    }
    return;
  }
  if (warp > W) return;

  // ---------------- consumers: 16 query rows per warp ----------------
  const int gq = lane >> 2, tq = lane & 3;
  const int G = p.G, R = p.R, T = a.T;
  int stage = 0;
  uint32_t phase = 0;
  bool fail = false;
  int b = 0;
  Seg sg;
  auto cta_of = [&](long long xx) { return split_cta_of(s_start, nct, xx); };
  for (long long x = start; !fail && next_seg(x, end, b, a, s_len, s_cum, sg); x = sg.ustart + sg.t1) {
    const uint64_t vis = tree_tiles_visible(a, sg.qt);
    const int row0 = sg.qt * p.rpt + warp * 16;
    const int ra = row0 + gq, rb = ra + 8;
    const int node_a = ra < R ? ra / G : -1, node_b = rb < R ? rb / G : -1;
    const __nv_bfloat16* qa = node_a >= 0 ? a.q + ((static_cast<size_t>(sg.b) * T + node_a) * a.Hq + sg.g * G + ra % G) * D : nullptr;
    const __nv_bfloat16* qb = node_b >= 0 ? a.q + ((static_cast<size_t>(sg.b) * T + node_b) * a.Hq + sg.g * G + rb % G) * D : nullptr;
    uint32_t qf[D / 16][4];
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      qf[kk][0] = qa ? ld_u32(qa + kk * 16 + 2 * tq) : 0u;
      qf[kk][1] = qb ? ld_u32(qb + kk * 16 + 2 * tq) : 0u;
      qf[kk][2] = qa ? ld_u32(qa + kk * 16 + 8 + 2 * tq) : 0u;
      qf[kk][3] = qb ? ld_u32(qb + kk * 16 + 8 + 2 * tq) : 0u;
    }
    float o[D / 8][4];
#pragma unroll
    for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;

    for (int t = sg.t0; t < sg.t1; ++t) {
      const bool tree = t >= sg.nc;
      const int j = t - sg.nc;
      if (tree && !((vis >> j) & 1ull)) continue;
      if (!tc::mbar_wait(full + stage, phase)) { fail = true; break; }
      const uint32_t tK = smem_u32(smem + stage * STAGE), tV = tK + HALF;
      const int k0 = tree ? j * KB : t * KB;
      const int valid = min(KB, (tree ? T : s_len[sg.b]) - k0);
      uint32_t wa0 = 0xffffffffu, wa1 = 0xffffffffu, wb0 = 0xffffffffu, wb1 = 0xffffffffu;
      if (tree) {
        const int w0 = 2 * j, mw = a.tr.mask_words;
        wa0 = node_a >= 0 ? a.tr.mask[static_cast<size_t>(node_a) * mw + w0] : 0u;
        wb0 = node_b >= 0 ? a.tr.mask[static_cast<size_t>(node_b) * mw + w0] : 0u;
        wa1 = (node_a >= 0 && w0 + 1 < mw) ? a.tr.mask[static_cast<size_t>(node_a) * mw + w0 + 1] : 0u;
        wb1 = (node_b >= 0 && w0 + 1 < mw) ? a.tr.mask[static_cast<size_t>(node_b) * mw + w0 + 1] : 0u;
      }
      const bool active = __any_sync(0xffffffffu, (wa0 | wa1 | wb0 | wb1) != 0u) && row0 < R;
      if (active) {
        // the tile in two halves of 32 keys, each an online-softmax update
#pragma unroll
        for (int hk = 0; hk < 2; ++hk) {
          constexpr int HK = KB / 2;
          float s[HK / 8][4];
#pragma unroll
          for (int nt = 0; nt < HK / 8; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
          for (int np = 0; np < HK / 16; ++np) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const int mat = lane >> 3, rr = lane & 7;
              uint32_t b0, b1, b2, b3;
              ldsm_x4(tile_addr(tK, hk * HK + np * 16 + (mat >> 1) * 8 + rr, kk * 2 + (mat & 1)), b0, b1, b2, b3);
              mma_bf16(s[2 * np], qf[kk], b0, b1);
              mma_bf16(s[2 * np + 1], qf[kk], b2, b3);
            }
          }
          const uint32_t wa = hk ? wa1 : wa0, wb = hk ? wb1 : wb0;
          float mx_a = -INFINITY, mx_b = -INFINITY;
#pragma unroll
          for (int nt = 0; nt < HK / 8; ++nt) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int kh = nt * 8 + 2 * tq + e;  // key within the half
              const bool in = hk * HK + kh < valid;
              const bool va = in && ((wa >> kh) & 1u);
              const bool vb = in && ((wb >> kh) & 1u);
              s[nt][e] = va ? s[nt][e] * a.scale_log2 : -INFINITY;
              s[nt][2 + e] = vb ? s[nt][2 + e] * a.scale_log2 : -INFINITY;
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
          for (int nt = 0; nt < HK / 8; ++nt) {
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
          // O += P V.  Keys past `valid` may hold anything (cache rows beyond
          // kv_len, another request's tree rows), so their V values are zeroed
          // in the fragments: a zero probability times a non-finite value is NaN.
#pragma unroll
          for (int kk = 0; kk < HK / 16; ++kk) {
            uint32_t pa[4];
            pa[0] = pack_bf16(s[2 * kk][0], s[2 * kk][1]);
            pa[1] = pack_bf16(s[2 * kk][2], s[2 * kk][3]);
            pa[2] = pack_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1]);
            pa[3] = pack_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3]);
            const int kA = hk * HK + kk * 16 + 2 * tq, kB = kA + 8;
            const uint32_t mA = (kA < valid ? 0x0000FFFFu : 0u) | (kA + 1 < valid ? 0xFFFF0000u : 0u);
            const uint32_t mB = (kB < valid ? 0x0000FFFFu : 0u) | (kB + 1 < valid ? 0xFFFF0000u : 0u);
#pragma unroll
            for (int dp = 0; dp < D / 16; ++dp) {
              const int mat = lane >> 3, rr = lane & 7;
              uint32_t b0, b1, b2, b3;
              ldsm_x4_t(tile_addr(tV, hk * HK + kk * 16 + (mat & 1) * 8 + rr, dp * 2 + (mat >> 1)), b0, b1, b2, b3);
              mma_bf16(o[2 * dp], pa, b0 & mA, b1 & mB);
              mma_bf16(o[2 * dp + 1], pa, b2 & mA, b3 & mB);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(empty + stage);
      if (++stage == kStages) { stage = 0; phase ^= 1; }
    }
    if (fail) break;

    // ---- this segment's result: final, or a partial for the combine launch ----
    l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
    l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);
    const int c_first = cta_of(sg.ustart);
    const int nparts = cta_of(sg.uend - 1) - c_first + 1;
    const int hq_base = sg.g * G;
    if (nparts == 1) {
      if (node_a >= 0) {
        const float inv = 1.f / l_a;
        float* dst = a.out + ((static_cast<size_t>(sg.b) * T + node_a) * a.Hq + hq_base + ra % G) * D;
#pragma unroll
        for (int dn = 0; dn < D / 8; ++dn)
          *reinterpret_cast<float2*>(dst + dn * 8 + 2 * tq) = make_float2(o[dn][0] * inv, o[dn][1] * inv);
        if (tq == 0 && !(l_a > 0.f) && a.dev_status) atomicOr(a.dev_status + sg.b, MEDUSA_DEV_NAN);
      }
      if (node_b >= 0) {
        const float inv = 1.f / l_b;
        float* dst = a.out + ((static_cast<size_t>(sg.b) * T + node_b) * a.Hq + hq_base + rb % G) * D;
#pragma unroll
        for (int dn = 0; dn < D / 8; ++dn)
          *reinterpret_cast<float2*>(dst + dn * 8 + 2 * tq) = make_float2(o[dn][2] * inv, o[dn][3] * inv);
        if (tq == 0 && !(l_b > 0.f) && a.dev_status) atomicOr(a.dev_status + sg.b, MEDUSA_DEV_NAN);
      }
      continue;
    }
    const int slot = blockIdx.x * 2 + (start >= sg.ustart ? 0 : 1);
    const size_t prow = static_cast<size_t>(slot) * p.rpt + warp * 16;
    float* da = a.ws.o_part + (prow + gq) * D;
    float* db = a.ws.o_part + (prow + gq + 8) * D;
#pragma unroll
    for (int dn = 0; dn < D / 8; ++dn) {
      *reinterpret_cast<float2*>(da + dn * 8 + 2 * tq) = make_float2(o[dn][0], o[dn][1]);
      *reinterpret_cast<float2*>(db + dn * 8 + 2 * tq) = make_float2(o[dn][2], o[dn][3]);
    }
    if (tq == 0) {
      a.ws.ml_part[prow + gq] = make_float2(m_a, l_a);
      a.ws.ml_part[prow + gq + 8] = make_float2(m_b, l_b);
    }
  }
  if (fail && lane == 0 && a.dev_status) atomicOr(a.dev_status + sg.b, MEDUSA_DEV_TIMEOUT);
}

// ---------------------------------------------------------------------------
// bf16 path on the tcgen05 tensor cores.  Same split of key tiles, same
// partial format.  Per CTA: warps 0-3 run the softmax (thread = query row of
// the 128-row tile), warp 4 streams Q (once per segment) and K/V tiles with
// TMA, warp 5 issues the MMAs and owns TMEM:
//   S = Q K^T (M 128, N 64 keys, K = D) into TMEM columns [0, 64) or
//   [64, 128) (two buffers: S of the next tile is computed while the softmax
//   works on this one);
//   the softmax threads read their S row, mask it (kv_len / cached tree bits),
//   exponentiate against a running maximum and write P (bf16) into the K half
//   of the tile's stage, which S no longer needs;
//   O += P V (M 128, N = D, K 64 keys; V read as an MN-major operand) into
//   TMEM columns [128, 128 + D).
// A softmax thread rescales its O row only when its maximum grows by more
// than 2^8 (P stays below 256 otherwise), which random or trained scores
// almost never need after the first tile; it then first waits for PV of the
// previous tile to complete (nothing else can be writing O at that point).
// ---------------------------------------------------------------------------
constexpr int kTcStages = 2;
constexpr int kTcThreads = 192;       // warps 0-3 softmax, 4 producer, 5 MMA
constexpr float kRescaleLog2 = 8.f;

template <int D>
struct TcLayout {
  static constexpr uint32_t NSUB = D / 64;
  static constexpr uint32_t Q_BYTES = NSUB * 128 * 128;  // [NSUB][128 rows][128 B]
  static constexpr uint32_t HALF = NSUB * 64 * 128;      // K or V: [NSUB][64 keys][128 B]
  static constexpr uint32_t STAGE = 2 * HALF;
  static constexpr uint32_t OFF_KV = Q_BYTES;
  static constexpr uint32_t P_BYTES = 128 * 128;         // [128 rows][64 keys] bf16
  // P goes into the K half of its tile's stage when that holds 128 rows
  static constexpr bool P_IN_K = HALF >= P_BYTES;
  static constexpr uint32_t OFF_P = OFF_KV + kTcStages * STAGE;  // two own buffers otherwise
  static constexpr uint32_t OFF_BAR = OFF_P + (P_IN_K ? 0 : 2 * P_BYTES);
  static constexpr uint32_t BYTES = OFF_BAR + 256;
  static constexpr uint32_t TMEM_O = 128;                 // first O column
  // P of the ti-th tile (stage st): the stage's K half, or buffer ti % 2
  __device__ static uint32_t p_off(int st, int ti) { return P_IN_K ? OFF_KV + st * STAGE : OFF_P + (ti & 1) * P_BYTES; }
};


// Visible tiles of a segment (cache tiles always, tree tiles per the mask).
__device__ inline int seg_visible_tiles(const Seg& sg, uint64_t vis) {
  int n = 0;
  for (int t = sg.t0; t < sg.t1; ++t) n += (t < sg.nc) || ((vis >> (t - sg.nc)) & 1ull);
  return n;
}

template <int D>
__global__ void __launch_bounds__(kTcThreads) tree_attn_tc_kernel(
    const __grid_constant__ CUtensorMap tm_kc, const __grid_constant__ CUtensorMap tm_vc,
    const __grid_constant__ CUtensorMap tm_kt, const __grid_constant__ CUtensorMap tm_vt,
    const __grid_constant__ CUtensorMap tm_q, AttnArgs a) {
  using Lay = TcLayout<D>;
  constexpr int NSUB = Lay::NSUB;
  extern __shared__ __align__(1024) unsigned char attn_tc_smem[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(attn_tc_smem) + 1023) & ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + Lay::OFF_BAR);
  uint64_t* kv_full = bar;                 // [kTcStages]
  uint64_t* kv_empty = bar + kTcStages;    // [kTcStages]
  uint64_t* q_full = bar + 2 * kTcStages;
  uint64_t* q_empty = q_full + 1;
  uint64_t* s_full = q_full + 2;   // [2]: one per S buffer (tile parity)
  uint64_t* p_full = q_full + 4;   // [2]: one per tile parity
  uint64_t* o_full = q_full + 6;
  uint64_t* o_free = q_full + 7;
  uint64_t* mma_done = q_full + 8;
  uint64_t* pv_done = q_full + 9;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(q_full + 10);
  __shared__ int s_len[MEDUSA_MAX_BATCH];
  __shared__ long long s_cum[MEDUSA_MAX_BATCH + 1];
  __shared__ long long s_start[kMaxSplit + 1];
  __shared__ uint64_t s_vis[kMaxVisTiles];
  __shared__ volatile int s_fail;

  const AttnPlan& p = a.p;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    s_fail = 0;
    for (int st = 0; st < kTcStages; ++st) {
      tc::mbar_init(kv_full + st, 1);
      tc::mbar_init(kv_empty + st, 1);
    }
    tc::mbar_init(q_full, 1);
    tc::mbar_init(q_empty, 1);
    tc::mbar_init(s_full, 1);
    tc::mbar_init(s_full + 1, 1);
    tc::mbar_init(pv_done, 1);
    tc::mbar_init(p_full, 4);
    tc::mbar_init(p_full + 1, 4);
    tc::mbar_init(o_full, 1);
    tc::mbar_init(o_free, 4);
    tc::mbar_init(mma_done, 1);
    tc::fence_mbar_init();
    tc::prefetch_tmap(&tm_kc);
    tc::prefetch_tmap(&tm_vc);
    tc::prefetch_tmap(&tm_kt);
    tc::prefetch_tmap(&tm_vt);
    tc::prefetch_tmap(&tm_q);
  }
  if (warp == 5) tc::tmem_alloc(tmem_slot, 256);
  if (a.vis_known)
    for (int i = threadIdx.x; i < p.n_qt; i += blockDim.x) s_vis[i] = a.vis[i];
  pdl_wait();
  for (int b = threadIdx.x; b < a.B; b += blockDim.x) s_len[b] = min(max(a.kv_len[b], 0), a.Lmax);
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t taddr = *tmem_slot;
  if (threadIdx.x == 0) {
    long long c = 0;
    const int upb = a.Hkv * p.n_qt;
    for (int b = 0; b < a.B; ++b) {
      s_cum[b] = c;
      c += static_cast<long long>(upb) * (cdiv(s_len[b], KB) + p.ntt);
    }
    s_cum[a.B] = c;
  }
  __syncthreads();
  pdl_trigger();
  const long long total = s_cum[a.B];
  const int nct = static_cast<int>(min(static_cast<long long>(gridDim.x), total));
  build_split(s_start, total, nct);
  __syncthreads();
  const bool active_cta = static_cast<int>(blockIdx.x) < nct;
  const long long start = active_cta ? s_start[blockIdx.x] : 0;
  const long long end = active_cta ? s_start[blockIdx.x + 1] : 0;
  const int G = p.G;

  if (warp == 4) {
    // ---------------- producer (whole warp walks the segments, lane 0 issues) ----------------
    int ti = 0, si = 0;
    bool ok = true;
    int b = 0;
    Seg sg;
    for (long long x = start; ok && next_seg(x, end, b, a, s_len, s_cum, sg); x = sg.ustart + sg.t1) {
      const uint64_t vis = (a.vis_known ? s_vis[sg.qt] : tree_tiles_visible(a, sg.qt));
      if (seg_visible_tiles(sg, vis) == 0) continue;
      if (lane == 0) {
        ok = !s_fail && tc::mbar_wait(q_empty, (si & 1) ^ 1);
        if (ok) {
          tc::mbar_expect_tx(q_full, Lay::Q_BYTES);
          const int node0 = sg.qt * p.rpt / G;
#pragma unroll
          for (int h = 0; h < NSUB; ++h)
            tc::tma_load_3d(smem_u32(smem + h * 16384), &tm_q, 64 * h, sg.g * G, sg.b * a.T + node0, q_full);
        }
        for (int t = sg.t0; ok && t < sg.t1; ++t) {
          const bool tree = t >= sg.nc;
          const int j = t - sg.nc;
          if (tree && !((vis >> j) & 1ull)) continue;
          const int st = ti % kTcStages;
          if (!tc::mbar_wait(kv_empty + st, ((ti / kTcStages) & 1) ^ 1)) { ok = false; break; }
          tc::mbar_expect_tx(kv_full + st, Lay::STAGE);
          const uint32_t sk = smem_u32(smem + Lay::OFF_KV + st * Lay::STAGE), sv = sk + Lay::HALF;
#pragma unroll
          for (int h = 0; h < NSUB; ++h) {
            if (!tree) {
              const int z = sg.b * a.Hkv + sg.g;
              tc::tma_load_3d(sk + h * 8192, &tm_kc, 64 * h, t * KB, z, kv_full + st);
              tc::tma_load_3d(sv + h * 8192, &tm_vc, 64 * h, t * KB, z, kv_full + st);
            } else {
              const int z = sg.b * a.T + j * KB;
              tc::tma_load_3d(sk + h * 8192, &tm_kt, 64 * h, sg.g, z, kv_full + st);
              tc::tma_load_3d(sv + h * 8192, &tm_vt, 64 * h, sg.g, z, kv_full + st);
            }
          }
          ++ti;
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      ++si;
    }
    if (lane == 0) {
      // every issued copy must have landed before the CTA's shared memory goes away
      for (int i = 0; i < min(ti, kTcStages); ++i) {
        const int k = ti - 1 - i;
        ok &= tc::mbar_wait(kv_full + (k % kTcStages), static_cast<uint32_t>((k / kTcStages) & 1));
      }
      if (si > 0) ok &= tc::mbar_wait(q_full, static_cast<uint32_t>((si - 1) & 1));
      if (!ok) s_fail = 1;
    }
  } else if (warp == 5) {
    // ---------------- MMA issuer (whole warp walks the segments, lane 0 issues) ----------------
    constexpr uint32_t idesc_s = tc::idesc_bf16_f32(128, KB);
    constexpr uint32_t idesc_o = tc::idesc_bf16_f32_bmn(128, D);
    const uint32_t tS = taddr, tO = taddr + Lay::TMEM_O;
    // base descriptors stepped with desc_add: the integer work between MMAs is what
    // bounds their issue rate from one thread
    const uint64_t dq = tc::smem_desc_sw128(smem_u32(smem));
    const uint64_t dkv0 = tc::smem_desc_sw128(smem_u32(smem + Lay::OFF_KV));
    const uint64_t dv0 = tc::smem_desc_sw128_lbo_sbo(smem_u32(smem + Lay::OFF_KV + Lay::HALF), 8192, 1024);
    int ti = 0, si = 0;
    bool ok = true;
    int b = 0;
    Seg sg;
    for (long long x = start; ok && next_seg(x, end, b, a, s_len, s_cum, sg); x = sg.ustart + sg.t1) {
      const uint64_t vis = (a.vis_known ? s_vis[sg.qt] : tree_tiles_visible(a, sg.qt));
      const int nt = seg_visible_tiles(sg, vis);
      if (nt == 0) continue;
      if (lane == 0) {
        ok = tc::mbar_wait(q_full, si & 1);
        int npv = 0, prev = -1;
        // O += P V for tile index `tix` (stage st)
        auto issue_pv = [&](int st, int tix) {
          if (!tc::mbar_wait(p_full + (tix & 1), (tix >> 1) & 1)) { ok = false; return; }
          if (npv == 0 && si > 0 && !tc::mbar_wait(o_free, (si - 1) & 1)) { ok = false; return; }
          tc::fence_after_sync();
          const uint64_t dp = tc::smem_desc_sw128(smem_u32(smem + Lay::p_off(st, tix)));
          const uint64_t dv = tc::desc_add(dv0, st * Lay::STAGE);
#pragma unroll
          for (int kk = 0; kk < KB / 16; ++kk)
            tc::mma_bf16(tO, tc::desc_add(dp, kk * 32), tc::desc_add(dv, kk * 2048), idesc_o, (npv | kk) != 0);
          tc::mma_commit(kv_empty + st);
          tc::mma_commit(pv_done);
          ++npv;
        };
        for (int k = 0; ok && k < nt; ++k) {
          const int st = ti % kTcStages;
          if (!tc::mbar_wait(kv_full + st, (ti / kTcStages) & 1)) { ok = false; break; }
          // S(ti) into buffer ti % 2: the softmax of tile ti-2 is done with it
          // (its P was waited for before PV(ti-2) was issued)
          tc::fence_after_sync();
          const uint64_t dk = tc::desc_add(dkv0, st * Lay::STAGE);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            tc::mma_bf16(tS + (ti & 1) * KB, tc::desc_add(dq, (kk >> 2) * 16384 + (kk & 3) * 32),
                         tc::desc_add(dk, (kk >> 2) * 8192 + (kk & 3) * 32), idesc_s, kk != 0);
          tc::mma_commit(s_full + (ti & 1));
          if (k == nt - 1) tc::mma_commit(q_empty);
          if (k > 0) {
            issue_pv(prev, ti - 1);
            if (!ok) break;
          }
          prev = st;
          ++ti;
        }
        if (ok) issue_pv(prev, ti - 1);
        if (ok) tc::mma_commit(o_full);
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      ++si;
    }
    if (lane == 0) {
      // TMEM is freed at the end: wait until every MMA issued here has completed
      tc::mma_commit(mma_done);
      if (!tc::mbar_wait(mma_done, 0)) ok = false;
      if (!ok) s_fail = 1;
    }
    __syncwarp();
  } else {
    // ---------------- softmax / epilogue: thread = query row ----------------
    const int row = threadIdx.x;  // 0..127
    const uint32_t tl = taddr + (static_cast<uint32_t>(warp * 32) << 16);
    int ts = 0, so = 0;
    bool ok = true;
    int b = 0;
    Seg sg;
    auto cta_of = [&](long long xx) { return split_cta_of(s_start, nct, xx); };
    for (long long x = start; next_seg(x, end, b, a, s_len, s_cum, sg); x = sg.ustart + sg.t1) {
      const uint64_t vis = (a.vis_known ? s_vis[sg.qt] : tree_tiles_visible(a, sg.qt));
      const int nt = ok ? seg_visible_tiles(sg, vis) : 0;
      const int r = sg.qt * p.rpt + row;
      const bool vrow = row < p.rpt && r < p.R;
      const int node = vrow ? r / G : 0;
      float m_used = -INFINITY, l = 0.f;
      int k = 0;
      for (int t = sg.t0; ok && t < sg.t1; ++t) {
        const bool tree = t >= sg.nc;
        const int j = t - sg.nc;
        if (tree && !((vis >> j) & 1ull)) continue;
        const int st = ts % kTcStages;
        const int k0 = tree ? j * KB : t * KB;
        const int vc = min(KB, (tree ? a.T : s_len[sg.b]) - k0);  // keys of this tile that exist
        uint32_t w0 = 0xffffffffu, w1 = 0xffffffffu;
        if (tree) {
          const int mw = a.tr.mask_words;
          w0 = vrow ? a.tr.mask[static_cast<size_t>(node) * mw + 2 * j] : 0u;
          w1 = (vrow && 2 * j + 1 < mw) ? a.tr.mask[static_cast<size_t>(node) * mw + 2 * j + 1] : 0u;
        }
        ok = __all_sync(0xffffffffu, tc::mbar_wait(s_full + (ts & 1), (ts >> 1) & 1));
        if (!ok) break;
        tc::fence_after_sync();
        float sv[64];
        {
          float h0[32], h1[32];
          tc::tmem_ld32(tl + (ts & 1) * KB, h0);
          tc::tmem_ld32(tl + (ts & 1) * KB + 32, h1);
#pragma unroll
          for (int e = 0; e < 32; ++e) { sv[e] = h0[e]; sv[32 + e] = h1[e]; }
        }
        // keys this row keeps (existing, and visible in the tree); raw scores of
        // the others become -inf.  Most tiles keep every key of every row.
        uint64_t km = 0;
        if (vrow) {
          km = vc >= KB ? ~0ull : ((1ull << vc) - 1);
          if (tree) km &= (static_cast<uint64_t>(w1) << 32) | w0;
        }
        if (!__all_sync(0xffffffffu, km == ~0ull)) {
#pragma unroll
          for (int e = 0; e < 64; ++e) sv[e] = ((km >> e) & 1ull) ? sv[e] : -INFINITY;
        }
        // tile maximum by a tree of pairwise maxima (raw scores: the scale is > 0)
        float mx[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) mx[e] = fmaxf(sv[e], sv[e + 32]);
#pragma unroll
        for (int h = 16; h >= 1; h >>= 1)
#pragma unroll
          for (int e = 0; e < h; ++e) mx[e] = fmaxf(mx[e], mx[e + h]);
        const float tm = mx[0] == -INFINITY ? -INFINITY : mx[0] * a.scale_log2;
        // lazy rescale: a row moves its exponent base only when its maximum grows
        // by more than 2^8; TMEM loads/stores are warp-collective, so the warp
        // rescales together when any of its rows needs it (factor 1 elsewhere)
        const bool grow = tm > m_used + kRescaleLog2 || (m_used == -INFINITY && tm > -INFINITY);
        const bool needs_o = grow && k > 0 && m_used > -INFINITY;
        if (__any_sync(0xffffffffu, needs_o)) {
          // PV of the previous tile must be complete before O is rewritten
          ok = __all_sync(0xffffffffu, tc::mbar_wait(pv_done, (ts - 1) & 1));
          if (!ok) break;
          tc::fence_after_sync();
          const float al = needs_o ? exp2f(m_used - tm) : 1.f;
#pragma unroll 1
          for (int c = 0; c < D; c += 32) {
            float ov[32];
            tc::tmem_ld32(tl + Lay::TMEM_O + c, ov);
#pragma unroll
            for (int e = 0; e < 32; ++e) ov[e] *= al;
            tc::tmem_st32(tl + Lay::TMEM_O + c, ov);
          }
          tc::tmem_st_wait();
          l *= al;
        }
        if (grow) m_used = tm;
        // P = 2^(s * scale - m) as bf16, 128-byte swizzled, keys along K
        unsigned char* prow = smem + Lay::p_off(st, ts) + row * 128;
        const bool any = m_used > -INFINITY;
        const float nb = any ? -m_used : 0.f;
        float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t pk[4];
#pragma unroll
          for (int q2 = 0; q2 < 4; ++q2) {
            float p0 = ex2_approx(fmaf(sv[c * 8 + 2 * q2], a.scale_log2, nb));
            float p1 = ex2_approx(fmaf(sv[c * 8 + 2 * q2 + 1], a.scale_log2, nb));
            p0 = any ? p0 : 0.f;
            p1 = any ? p1 : 0.f;
            ps[q2] += p0 + p1;
            __nv_bfloat162 v2 = __floats2bfloat162_rn(p0, p1);
            pk[q2] = *reinterpret_cast<uint32_t*>(&v2);
          }
          *reinterpret_cast<uint4*>(prow + ((c ^ (row & 7)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
        const float psum = (ps[0] + ps[1]) + (ps[2] + ps[3]);
        l += psum;
        if (vc < KB) {
          // keys past the end may hold anything: zero their V rows (P is 0 there,
          // and 0 times a non-finite value is NaN)
          unsigned char* vbase = smem + Lay::OFF_KV + st * Lay::STAGE + Lay::HALF;
          const int nrow = KB - vc, n16 = nrow * 8 * NSUB;
          for (int e = row; e < n16; e += 128) {
            const int h = e / (nrow * 8), rr = vc + (e / 8) % nrow, c = e % 8;
            *reinterpret_cast<uint4*>(vbase + h * 8192 + rr * 128 + c * 16) = make_uint4(0, 0, 0, 0);
          }
        }
        tc::fence_proxy_async_smem();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(p_full + (ts & 1));
        ++ts;
        ++k;
      }
      // ---- segment result: final rows, or a partial for the combine launch ----
      if (nt > 0 && ok) ok = __all_sync(0xffffffffu, tc::mbar_wait(o_full, so & 1));
      if (!ok) break;
      const int c_first = cta_of(sg.ustart);
      const bool whole = cta_of(sg.uend - 1) == c_first;
      float* dst = nullptr;
      float scale = 1.f;
      if (whole && vrow) {
        dst = a.out + ((static_cast<size_t>(sg.b) * a.T + node) * a.Hq + sg.g * G + r % G) * D;
        scale = 1.f / l;
        if (!(l > 0.f) && a.dev_status) atomicOr(a.dev_status + sg.b, MEDUSA_DEV_NAN);
      } else if (!whole && row < p.rpt) {
        const int slot = blockIdx.x * 2 + (start >= sg.ustart ? 0 : 1);
        const size_t prw = static_cast<size_t>(slot) * p.rpt + row;
        dst = a.ws.o_part + prw * D;
        a.ws.ml_part[prw] = make_float2(m_used, l);
      }
      if (nt > 0) {
        tc::fence_after_sync();
#pragma unroll 1
        for (int c = 0; c < D; c += 32) {
          float ov[32];
          tc::tmem_ld32(tl + Lay::TMEM_O + c, ov);
          if (dst)
#pragma unroll
            for (int e = 0; e < 32; e += 4)
              *reinterpret_cast<float4*>(dst + c + e) =
                  make_float4(ov[e] * scale, ov[e + 1] * scale, ov[e + 2] * scale, ov[e + 3] * scale);
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(o_free);
        ++so;
      } else if (dst) {
        for (int e = 0; e < D; e += 4) *reinterpret_cast<float4*>(dst + e) = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    if (!ok) s_fail = 1;
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 5) tc::tmem_dealloc(taddr, 256);
  if (threadIdx.x == 0 && s_fail && a.dev_status)
    for (int b = 0; b < a.B; ++b) atomicOr(a.dev_status + b, MEDUSA_DEV_TIMEOUT);
}

// Merge the partials of every head that spans several CTAs: one warp per
// (head unit, query row), parts in CTA order.  The split is recomputed from
// kv_len exactly as the attention launch made it.
template <int D>
__global__ void __launch_bounds__(256) attn_combine_kernel(AttnArgs a, int attn_ctas) {
  __shared__ int s_len[MEDUSA_MAX_BATCH];
  __shared__ long long s_cum[MEDUSA_MAX_BATCH + 1];
  __shared__ long long s_start[kMaxSplit + 1];
  const AttnPlan& p = a.p;
  pdl_wait();
  pdl_trigger();
  for (int b = threadIdx.x; b < a.B; b += blockDim.x) s_len[b] = min(max(a.kv_len[b], 0), a.Lmax);
  __syncthreads();
  if (threadIdx.x == 0) {
    long long c = 0;
    const int upb = a.Hkv * p.n_qt;
    for (int b = 0; b < a.B; ++b) {
      s_cum[b] = c;
      c += static_cast<long long>(upb) * (cdiv(s_len[b], KB) + p.ntt);
    }
    s_cum[a.B] = c;
  }
  __syncthreads();
  const long long total = s_cum[a.B];
  const int nct = static_cast<int>(min(static_cast<long long>(attn_ctas), total));
  build_split(s_start, total, nct);
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (gw >= p.units * p.rpt) return;
  const int unit = gw / p.rpt, row = gw % p.rpt;
  const int qt = unit % p.n_qt, g = (unit / p.n_qt) % a.Hkv, b = unit / (p.n_qt * a.Hkv);
  const int r = qt * p.rpt + row;
  if (r >= p.R) return;
  const int cost = cdiv(s_len[b], KB) + p.ntt;
  const long long ustart = s_cum[b] + static_cast<long long>(g * p.n_qt + qt) * cost;
  const int c_first = split_cta_of(s_start, nct, ustart);
  const int nparts = split_cta_of(s_start, nct, ustart + cost - 1) - c_first + 1;
  if (nparts == 1) return;  // written by the attention launch
  auto part_row = [&](int q) -> size_t {
    const int c = c_first + q;
    return static_cast<size_t>(c * 2 + (s_start[c] >= ustart ? 0 : 1)) * p.rpt + row;
  };
  // running max and denominator over the parts (lanes take parts)
  float M = -INFINITY;
  for (int q = lane; q < nparts; q += 32) {
    const float2 ml = __ldcg(a.ws.ml_part + part_row(q));
    if (ml.y > 0.f) M = fmaxf(M, ml.x);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  constexpr int PER = D / 32;  // columns per lane
  float acc[PER] = {};
  float den = 0.f;
  for (int q0 = 0; q0 < nparts; q0 += 32) {
    float wq = 0.f;
    size_t prq = 0;
    if (q0 + lane < nparts) {
      prq = part_row(q0 + lane);
      const float2 ml = __ldcg(a.ws.ml_part + prq);
      if (ml.y > 0.f) {
        wq = exp2f(ml.x - M);
        den = fmaf(wq, ml.y, den);
      }
    }
    const int nq = min(32, nparts - q0);
    constexpr int UQ = 8;
    for (int j0 = 0; j0 < nq; j0 += UQ) {
      float v[UQ][PER];
      float wj[UQ];
#pragma unroll
      for (int j = 0; j < UQ; ++j) {
        wj[j] = __shfl_sync(0xffffffffu, wq, (j0 + j) & 31);
        const size_t pr = __shfl_sync(0xffffffffu, prq, (j0 + j) & 31);
        if (j0 + j < nq) {
          const float* src = a.ws.o_part + pr * D + lane * PER;
          if constexpr (PER == 4) {
            const float4 t = __ldcg(reinterpret_cast<const float4*>(src));
            v[j][0] = t.x; v[j][1] = t.y; v[j][2] = t.z; v[j][3] = t.w;
          } else {
            const float2 t = __ldcg(reinterpret_cast<const float2*>(src));
            v[j][0] = t.x; v[j][1] = t.y;
          }
        }
      }
#pragma unroll
      for (int j = 0; j < UQ; ++j)
        if (j0 + j < nq)
#pragma unroll
          for (int e = 0; e < PER; ++e) acc[e] = fmaf(wj[j], v[j][e], acc[e]);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
  const int node = r / p.G;
  float* dst = a.out + ((static_cast<size_t>(b) * a.T + node) * a.Hq + g * p.G + r % p.G) * D + lane * PER;
  const float inv = 1.f / den;
  if constexpr (PER == 4) {
    *reinterpret_cast<float4*>(dst) = make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
  } else {
    *reinterpret_cast<float2*>(dst) = make_float2(acc[0] * inv, acc[1] * inv);
  }
  if (lane == 0 && !(den > 0.f) && a.dev_status) atomicOr(a.dev_status + b, MEDUSA_DEV_NAN);
}

// Rotary position embedding of the tree's queries and keys (rotate-half form,
// Su et al., "RoFormer", 2021): for d < D/2 the pair (x[d], x[d + D/2]) turns by
// position * theta^(-2d/D).  One CTA per tree node; the D/2 angles are computed
// once per node in double precision (positions reach the tens of thousands) and
// shared by every head of the node.
template <typename T>
__global__ void __launch_bounds__(256) rope_kernel(const T* __restrict__ q, const T* __restrict__ k,
                                                   const int32_t* __restrict__ pos, int Hq, int Hkv, int D,
                                                   double log2_theta, T* __restrict__ q_out, T* __restrict__ k_out) {
  __shared__ float s_c[64], s_s[64];
  const size_t node = blockIdx.x;  // b * T + i
  const int half = D / 2;
  pdl_wait();
  pdl_trigger();
  if (static_cast<int>(threadIdx.x) < half) {
    const double ang = static_cast<double>(pos[node]) * exp2(-(2.0 * threadIdx.x / D) * log2_theta);
    double sn, cs;
    sincos(ang, &sn, &cs);
    s_c[threadIdx.x] = static_cast<float>(cs);
    s_s[threadIdx.x] = static_cast<float>(sn);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < (Hq + Hkv) * half; e += blockDim.x) {
    const int h = e / half, d = e % half;
    const T* src = h < Hq ? q + (node * Hq + h) * D : k + (node * Hkv + (h - Hq)) * D;
    T* dst = h < Hq ? q_out + (node * Hq + h) * D : k_out + (node * Hkv + (h - Hq)) * D;
    const float x0 = Elem<T>::to_f(src[d]), x1 = Elem<T>::to_f(src[d + half]);
    const float c = s_c[d], sn = s_s[d];
    dst[d] = Elem<T>::from_f(fmaf(x0, c, -x1 * sn));
    dst[d + half] = Elem<T>::from_f(fmaf(x1, c, x0 * sn));
  }
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
  pdl_wait();
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

// Bytes of the rotated queries and keys held ahead of the split partials in the workspace.
size_t rope_ws_bytes(int B, int T, int Hq, int Hkv, int D, int es) {
  return align_up(static_cast<size_t>(B) * T * Hq * D * es, 256) + align_up(static_cast<size_t>(B) * T * Hkv * D * es, 256);
}

MEDUSA_API size_t medusa_tree_attention_workspace_size(const medusa_tree* tree, int32_t B, int32_t Hq, int32_t Hkv,
                                                       int32_t D, int32_t Lmax, int32_t kv_len_hint,
                                                       medusa_dtype dtype) {
  if (!tree || B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv || Lmax < 0) return 0;
  if (D != 64 && D != 128) return 0;
  const size_t rope = rope_ws_bytes(B, tree->T, Hq, Hkv, D, dtype == MEDUSA_BF16 ? 2 : 4);
  if (dtype == MEDUSA_F32) return rope;
  AttnPlan p = plan_attn(tree->T, B, Hq, Hkv, Lmax, kv_len_hint, device_sm_count());
  return rope + carve_attn_ws(nullptr, p, D).bytes;
}

namespace {

template <int D>
int launch_attn_bf16(const medusa_tree* tree, const void* q, const void* k_new, const void* v_new,
                     const void* k_cache, const void* v_cache, const int32_t* kv_len, int B, int Hq, int Hkv,
                     int Lmax, float scale, float* out, const AttnPlan& p, const AttnWs& w, int32_t* dev_status,
                     cudaStream_t st) {
  const int T = tree->T;
  CUtensorMap kc, vc, kt, vt;
  const uint64_t rowb = static_cast<uint64_t>(D) * 2;
  const uint64_t lm = static_cast<uint64_t>(std::max(Lmax, 1));
  if (!make_tmap_bf16_3d(&kc, k_cache, D, lm, static_cast<uint64_t>(B) * Hkv, rowb, lm * rowb, KB, 1) ||
      !make_tmap_bf16_3d(&vc, v_cache, D, lm, static_cast<uint64_t>(B) * Hkv, rowb, lm * rowb, KB, 1) ||
      !make_tmap_bf16_3d(&kt, k_new, D, Hkv, static_cast<uint64_t>(B) * T, rowb, Hkv * rowb, 1, KB) ||
      !make_tmap_bf16_3d(&vt, v_new, D, Hkv, static_cast<uint64_t>(B) * T, rowb, Hkv * rowb, 1, KB))
    return MEDUSA_ERR_CUDA;
  AttnArgs a{};
  a.tr = tree->dev;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.kv_len = kv_len;
  a.out = out;
  a.ws = w;
  a.dev_status = dev_status;
  a.B = B;
  a.T = T;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.Lmax = Lmax;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.p = p;
  a.vis_known = 0;
  if (p.n_qt <= kMaxVisTiles) {
    const std::vector<uint64_t>& v = tree_tile_visibility(const_cast<medusa_tree*>(tree), p.G, p.rpt);
    for (int i = 0; i < p.n_qt; ++i) a.vis[i] = v[i];
    a.vis_known = 1;
  }
  if (128 % p.G == 0) {
    // tensor-core path: Q tiles of 128 rows (node, query head of the group) by TMA
    CUtensorMap tq;
    if (!make_tmap_bf16_3d(&tq, q, D, Hq, static_cast<uint64_t>(B) * T, rowb, static_cast<uint64_t>(Hq) * rowb, p.G,
                           128 / p.G))
      return MEDUSA_ERR_CUDA;
    const size_t smem = 1024 + TcLayout<D>::BYTES;
    auto k = tree_attn_tc_kernel<D>;
    if (!ensure_dyn_smem(k, smem))
      return MEDUSA_ERR_CUDA;
    if (launch_pdl(k, dim3(p.nctas), dim3(kTcThreads), smem, st, kc, vc, kt, vt, tq, a) != cudaSuccess) {
      (void)cudaGetLastError();
      return MEDUSA_ERR_CUDA;
    }
  } else {
    const size_t smem = 1024 + static_cast<size_t>(kStages) * 2 * (D / 64) * 8192 + 2 * kStages * 8;
    auto k = tree_attn_kernel<D>;
    if (!ensure_dyn_smem(k, smem))
      return MEDUSA_ERR_CUDA;
    if (launch_pdl(k, dim3(p.nctas), dim3((p.W + 1) * 32), smem, st, kc, vc, kt, vt, a) != cudaSuccess) {
      (void)cudaGetLastError();
      return MEDUSA_ERR_CUDA;
    }
  }
  MEDUSA_LAUNCH_CHECK();
  const long long warps = static_cast<long long>(p.units) * p.rpt;
  if (launch_pdl(attn_combine_kernel<D>, dim3(static_cast<unsigned>((warps + 7) / 8)), dim3(256), 0, st, a,
                 p.nctas) != cudaSuccess) {
    (void)cudaGetLastError();
    return MEDUSA_ERR_CUDA;
  }
  MEDUSA_LAUNCH_CHECK();
  return MEDUSA_OK;
}

}  // namespace

MEDUSA_API int medusa_tree_attention(const medusa_tree* tree, const void* q, const void* k_new, const void* v_new,
                                     const void* k_cache, const void* v_cache, const int32_t* kv_len,
                                     const int32_t* position_ids, int32_t B, int32_t Hq, int32_t Hkv, int32_t D,
                                     int32_t Lmax, int32_t kv_len_hint, float scale, int32_t rope, float rope_theta,
                                     medusa_dtype dtype, float* out, void* k_rot, void* ws, size_t ws_bytes,
                                     int32_t* dev_status, medusa_stream_t stream) {
  if (!tree || !q || !k_new || !v_new || !k_cache || !v_cache || !kv_len || !out) return MEDUSA_ERR_INVALID_ARG;
  if (B < 1 || B > MEDUSA_MAX_BATCH || Hq < 1 || Hkv < 1 || Lmax < 0 || Hq > 128) return MEDUSA_ERR_INVALID_ARG;
  if (dtype != MEDUSA_F32 && dtype != MEDUSA_BF16) return MEDUSA_ERR_INVALID_ARG;
  if (rope && (!position_ids || !(rope_theta > 1.f))) return MEDUSA_ERR_INVALID_ARG;
  if (Hq % Hkv != 0 || (D != 64 && D != 128)) return MEDUSA_ERR_UNSUPPORTED;
  const void* ptrs[] = {q, k_new, v_new, k_cache, v_cache, kv_len, out};
  for (const void* x : ptrs)
    if (!aligned16(x)) return MEDUSA_ERR_ALIGNMENT;
  const void* opt[] = {ws, dev_status, position_ids, k_rot};
  for (const void* x : opt)
    if (x && !aligned16(x)) return MEDUSA_ERR_ALIGNMENT;
  auto st = reinterpret_cast<cudaStream_t>(stream);
  const int T = tree->T;
  const int es = dtype == MEDUSA_BF16 ? 2 : 4;
  const size_t rope_bytes = rope_ws_bytes(B, T, Hq, Hkv, D, es);
  char* wsc = static_cast<char*>(ws);
  if (rope) {
    // q and k_new rotated at the tree's position ids into the workspace (k into
    // k_rot when the caller keeps the rotated keys, e.g. to commit them)
    if (!ws || ws_bytes < rope_bytes) return MEDUSA_ERR_WORKSPACE;
    void* q_r = wsc;
    void* k_r = k_rot ? k_rot : wsc + align_up(static_cast<size_t>(B) * T * Hq * D * es, 256);
    const double l2t = std::log2(static_cast<double>(rope_theta));
    cudaError_t e;
    if (dtype == MEDUSA_BF16)
      e = launch_pdl(rope_kernel<__nv_bfloat16>, dim3(B * T), dim3(256), 0, st, static_cast<const __nv_bfloat16*>(q),
                     static_cast<const __nv_bfloat16*>(k_new), position_ids, Hq, Hkv, D, l2t,
                     static_cast<__nv_bfloat16*>(q_r), static_cast<__nv_bfloat16*>(k_r));
    else
      e = launch_pdl(rope_kernel<float>, dim3(B * T), dim3(256), 0, st, static_cast<const float*>(q),
                     static_cast<const float*>(k_new), position_ids, Hq, Hkv, D, l2t, static_cast<float*>(q_r),
                     static_cast<float*>(k_r));
    if (e != cudaSuccess) {
      (void)cudaGetLastError();
      return MEDUSA_ERR_CUDA;
    }
    MEDUSA_LAUNCH_CHECK();
    q = q_r;
    k_new = k_r;
  }
  if (dtype == MEDUSA_F32) {
    const size_t smem = static_cast<size_t>(Lmax + T) * 4;
    if (smem > 200 * 1024) return MEDUSA_ERR_UNSUPPORTED;
    if (!ensure_dyn_smem(tree_attn_f32_kernel, smem))
      return MEDUSA_ERR_CUDA;
    if (launch_pdl(tree_attn_f32_kernel, dim3(B * T * Hq), dim3(128), smem, st, tree->dev,
                   static_cast<const float*>(q), static_cast<const float*>(k_new), static_cast<const float*>(v_new),
                   static_cast<const float*>(k_cache), static_cast<const float*>(v_cache), kv_len, Hq, Hkv, D, Lmax,
                   scale, out) != cudaSuccess) {
      (void)cudaGetLastError();
      return MEDUSA_ERR_CUDA;
    }
    MEDUSA_LAUNCH_CHECK();
    return MEDUSA_OK;
  }
  AttnPlan p = plan_attn(T, B, Hq, Hkv, Lmax, kv_len_hint, device_sm_count());
  AttnWs w = carve_attn_ws(wsc ? wsc + rope_bytes : nullptr, p, D);
  if (!ws || ws_bytes < rope_bytes + w.bytes) return MEDUSA_ERR_WORKSPACE;
  if (D == 128)
    return launch_attn_bf16<128>(tree, q, k_new, v_new, k_cache, v_cache, kv_len, B, Hq, Hkv, Lmax, scale, out, p, w,
                                 dev_status, st);
  return launch_attn_bf16<64>(tree, q, k_new, v_new, k_cache, v_cache, kv_len, B, Hq, Hkv, Lmax, scale, out, p, w,
                              dev_status, st);
}
