// Multi-row GEMV core: R consecutive weight rows dotted with nb activation rows.
//
// The weight matrix is streamed once from HBM with 16-byte non-allocating
// loads, lane l of a warp taking chunks l, l+32, ... of a row (every load
// instruction of a warp covers 512 contiguous bytes); the activations sit in
// shared memory.  Each lane accumulates partial dot products in fp32 and the
// warp reduces them with shuffles.
#pragma once

#include "common.cuh"

namespace medusa {

// Loads of one row group kept in flight per lane: R rows x U chunks.
template <typename T, int BMAX, int R, int U>
__device__ inline void gemv_rows(const T* __restrict__ W, size_t row0, int rows_valid, int H,
                                 const T* __restrict__ xs, int nb, float (&acc)[R][BMAX]) {
  constexpr int E = Elem<T>::kPer16B;
  const int lane = threadIdx.x & 31;
  const int nchunks = H / E;
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int b = 0; b < BMAX; ++b) acc[r][b] = 0.f;

  const T* wrow[R];
#pragma unroll
  for (int r = 0; r < R; ++r) wrow[r] = W + (row0 + (r < rows_valid ? r : 0)) * static_cast<size_t>(H);

  for (int c0 = lane; c0 < nchunks; c0 += 32 * U) {
    uint4 w[U][R];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = c0 + u * 32;
#pragma unroll
      for (int r = 0; r < R; ++r)
        w[u][r] = (c < nchunks) ? ld_stream16(wrow[r] + static_cast<size_t>(c) * E) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = c0 + u * 32;
      if (c >= nchunks) break;
      float wf[R][E];
#pragma unroll
      for (int r = 0; r < R; ++r) unpack16(w[u][r], wf[r], static_cast<T*>(nullptr));
#pragma unroll
      for (int b = 0; b < BMAX; ++b) {
        if (b < nb) {
          const uint4 xv = *reinterpret_cast<const uint4*>(xs + static_cast<size_t>(b) * H + static_cast<size_t>(c) * E);
          float xf[E];
          unpack16(xv, xf, static_cast<T*>(nullptr));
#pragma unroll
          for (int r = 0; r < R; ++r)
#pragma unroll
            for (int e = 0; e < E; ++e) acc[r][b] = fmaf(wf[r][e], xf[e], acc[r][b]);
        }
      }
    }
  }
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int b = 0; b < BMAX; ++b)
      if (b < nb) acc[r][b] = warp_sum(acc[r][b]);
}

// Copy nb activation rows of length H (16-byte chunks) into shared memory.
template <typename T>
__device__ inline void stage_rows(T* xs, const T* __restrict__ x, size_t row_stride, int nb, int H) {
  constexpr int E = Elem<T>::kPer16B;
  const int nch = H / E;
  for (int e = threadIdx.x; e < nb * nch; e += blockDim.x) {
    const int b = e / nch, c = e % nch;
    *reinterpret_cast<uint4*>(xs + static_cast<size_t>(b) * H + static_cast<size_t>(c) * E) =
        *reinterpret_cast<const uint4*>(x + b * row_stride + static_cast<size_t>(c) * E);
  }
}

// --------------------------------------------------------------------------
// Block-wide top-k over (value, id) pairs held in shared memory.
// Order: larger value first, equal values by lower id, NaN last (never
// selected ahead of a number).  Values are consumed (set to NaN).
// Each warp selects the top-k of its slice, then warp 0 merges the slices.
// Result written to out_v/out_i (k entries; missing entries -> -inf / -1).
// scratch_v/scratch_i: 8*k entries.  All threads of the block must call.
// --------------------------------------------------------------------------
__device__ inline void warp_topk_slice(float* v, const int* ids, int id_base, int n, int k,
                                       float* out_v, int* out_i, float missing_val) {
  const int lane = threadIdx.x & 31;
  for (int t = 0; t < k; ++t) {
    float bv = -INFINITY;
    int bi = 0x7fffffff, bp = -1;
    for (int j = lane; j < n; j += 32) {
      const float x = v[j];
      const int id = ids ? ids[j] : id_base + j;
      if (better(x, id, bv, bi)) { bv = x; bi = id; bp = j; }
    }
    // warp argmax carrying the position
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      const int op = __shfl_xor_sync(0xffffffffu, bp, o);
      if (better(ov, oi, bv, bi) || (bp < 0 && op >= 0)) { bv = ov; bi = oi; bp = op; }
    }
    if (lane == 0) {
      out_v[t] = bp >= 0 ? bv : missing_val;
      out_i[t] = bp >= 0 ? bi : -1;
      if (bp >= 0) v[bp] = __int_as_float(0x7fc00000);  // taken
    }
    __syncwarp();
  }
}

__device__ inline void block_topk(float* v, int* ids, int id_base, int n, int k, float* out_v, int* out_i,
                                  float* scratch_v, int* scratch_i) {
  const int warp = threadIdx.x >> 5;
  const int nw = blockDim.x >> 5;
  const int per = cdiv(n, nw);
  const int s0 = min(n, warp * per), s1 = min(n, s0 + per);
  // slices mark missing entries NaN so the merge never picks them
  warp_topk_slice(v + s0, ids ? ids + s0 : nullptr, id_base + s0, s1 - s0, k, scratch_v + warp * k,
                  scratch_i + warp * k, __int_as_float(0x7fc00000));
  __syncthreads();
  if (warp == 0) warp_topk_slice(scratch_v, scratch_i, 0, nw * k, k, out_v, out_i, -INFINITY);
  __syncthreads();
}

}  // namespace medusa
