// Tensor-core GEMM for every dense contraction of the drafting hot path:
// fc over tap rows, K/V injection, the block's Q/K/V, O, gate/up and down
// projections, and the shared LM head.
//
// D[M, N] = A[M, K] * B[N, K]^T with A = weights (output features along M,
// one or more stacked projections) and B = activations (tokens along N). The
// weight is always the 128-row M operand, so a batch-1 block (16 tokens) is a
// 128 x 16 MMA tile and all the bandwidth goes to streaming weights.
//
// One CTA = 6 warps:
//   warp 0     one thread issues TMA tile loads (128-byte swizzle) into a ring
//              of shared-memory stages, signalling `full` mbarriers;
//   warp 1     allocates tensor memory; one thread issues tcgen05.mma
//              (kind::f16, bf16 x bf16 -> fp32 in TMEM) and commits to the
//              `empty` barrier of each stage and to `tmem_full` per tile;
//   warps 2-5  the epilogue: tcgen05.ld of the accumulator (warp w reads TMEM
//              lanes 32*(w%4)..+31), then the fused epilogue.
// The accumulator is double-buffered in TMEM when it fits, so the epilogue of
// one work unit overlaps the MMAs of the next. CTAs are persistent and walk
// the work units round-robin.
//
// Split-K: the reduction is cut into ksplit chunks. Either the chunks of a
// tile form a thread-block cluster and reduce through distributed shared
// memory, or each chunk writes its fp32 partial tile to global memory and the
// last chunk to finish a tile (atomic counter) adds all partials in chunk
// order and runs the epilogue. The host fixes ksplit from the weight's shape
// alone for small batches, so a token's result does not depend on the batch
// it runs in; wider batches take a split chosen for throughput.
#include <stdio.h>

#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

namespace dfl {

template <int BN, bool DUAL, int STAGES, int EPI>
struct GemmTraits {
  static constexpr int kABytes = kTileM * kTileK * 2;  // 16 KiB
  static constexpr int kBBytes = BN * kTileK * 2;
  static constexpr int kStageBytes = kABytes * (DUAL ? 2 : 1) + kBBytes;
  static constexpr int kAcc = DUAL ? 2 : 1;
  static constexpr int kAccCols = BN * kAcc;
  static constexpr int kAccBufs = (kAccCols * 2 <= 512) ? 2 : 1;
  static constexpr int kTmemNeed = kAccCols * kAccBufs;
  static constexpr int kTmemCols = kTmemNeed <= 32 ? 32 : kTmemNeed <= 64 ? 64 : kTmemNeed <= 128 ? 128
                                                            : kTmemNeed <= 256 ? 256 : 512;
  static constexpr int kBarBytes = 8 * (2 * STAGES + 2 * kAccBufs + 1) + 16;
  // rope partner exchange (heads) / the chunk's bf16 outputs for candidate ranking (store bf16)
  static constexpr int kXchFloats = EPI == EPI_HEADS ? kTileM * 17 : EPI == EPI_STORE_BF16 ? 16 * (kTileM + 1) : 0;
  static constexpr int kRedFloats =
      (EPI == EPI_HEADS || EPI == EPI_RESID || EPI == EPI_STORE_F32) ? 4 * 16 : 0;  // per-warp sums of squares
  static constexpr int kMetaInts = EPI == EPI_HEADS ? 4 * BN : 0;  // per-token (pos, stream, segment end)
  static constexpr int kSmemBytes =
      1024 /*alignment slack*/ + STAGES * kStageBytes + kBarBytes + 4 * (kXchFloats + kRedFloats + kMetaInts) + 64;
  static constexpr uint32_t kIdesc = idesc_bf16_f32(kTileM, BN);
  // cluster split-K parks each CTA's fp32 partial in its (idle) stage memory
  static constexpr bool kClusterFits = kAcc * BN * kTileM * 4 <= STAGES * kStageBytes;
};

// ---------------------------------------------------------------- cluster helpers
__device__ __forceinline__ uint32_t gemm_cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void gemm_cluster_sync() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
// The two halves of a cluster barrier: a thread arrives once its reads of
// other CTAs' shared memory are done and waits before its CTA exits.
__device__ __forceinline__ void gemm_cluster_arrive() { asm volatile("barrier.cluster.arrive.release;" ::: "memory"); }
__device__ __forceinline__ void gemm_cluster_wait() { asm volatile("barrier.cluster.wait.acquire;" ::: "memory"); }
__device__ __forceinline__ uint32_t gemm_mapa(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ float gemm_ld_dsmem(uint32_t a) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
  return v;
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }

// Work-unit order. Global split-K: ((m_tile * ksplit + kc) * n_tiles + n_tile),
// so concurrent CTAs share weight slabs across n-tiles. Cluster split-K:
// (tile * ksplit + kc), the chunks of a tile being one cluster.
template <bool CLU>
__device__ __forceinline__ void decode_unit(const GemmArgs& a, int u, int& m_tile, int& kc, int& n_tile) {
  if constexpr (CLU) {
    kc = u % a.ksplit;
    const int tile = u / a.ksplit;
    m_tile = tile / a.n_tiles;
    n_tile = tile - m_tile * a.n_tiles;
  } else {
    n_tile = u % a.n_tiles;
    const int r = u / a.n_tiles;
    kc = r % a.ksplit;
    m_tile = r / a.ksplit;
  }
  m_tile += a.m_tile0;  // the weight's tile index
}

__device__ __forceinline__ int seg_of_tile(const GemmArgs& a, int m_tile) {
  int s = 0;
  while (s + 1 < a.n_aseg && m_tile >= a.a_seg_tile[s + 1]) ++s;
  return s;
}

// ---------------------------------------------------------------- epilogues

// Sum v[j] over the 32 lanes for all 16 j at once: four halving exchanges
// then one pairwise add (16 shuffles). Lane L (and L ^ 1) ends with the total
// of column j = 8*b4 + 4*b3 + 2*b2 + b1 of L's bits; the order of the
// additions is fixed.
__device__ __forceinline__ float warp_sum16(const float (&v)[16], int lane, int& j_out) {
  float a[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) a[j] = v[j];
#pragma unroll
  for (int h = 8, off = 16; h >= 1; h >>= 1, off >>= 1) {
    const bool up = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < h; ++i) {
      const float send = up ? a[i] : a[i + h];
      const float keep = up ? a[i + h] : a[i];
      a[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
  j_out = 8 * ((lane >> 4) & 1) + 4 * ((lane >> 3) & 1) + 2 * ((lane >> 2) & 1) + ((lane >> 1) & 1);
  return a[0] + __shfl_xor_sync(0xffffffffu, a[0], 1);
}
// v0 (and v1 for the dual GEMM) hold the accumulator of output feature
// m = m_tile*128 + row for tokens t = n0 + j, j = 0..15.
// ss_out[m_tile][t] = sum over the tile's 128 rows of sq (per column t of the
// chunk): warp partials by the transpose reduction, then the 4 warps in order.
__device__ __forceinline__ void publish_ss(const GemmArgs& a, const float (&sq)[16], int m_tile, int n0, int row,
                                           int q, int lane, float* red, int nvalid) {
  int jj;
  const float w = warp_sum16(sq, lane, jj);
  if ((lane & 1) == 0) red[q * 16 + jj] = w;
  named_bar_sync(1, 128);
  if (row < 16 && row < nvalid && n0 + row < a.N)
    a.epi.ss_out[static_cast<int64_t>(m_tile) * a.epi.ss_ld + n0 + row] =
        ((red[row] + red[16 + row]) + red[32 + row]) + red[48 + row];
  named_bar_sync(1, 128);  // red reusable by the next chunk
}

// Heads-epilogue operands of one warp's columns of a 16-column chunk
// (columns q, q + 4, q + 8, q + 12 of warp q; lane l holds features l + 32i):
// each column's position, stream and segment end, the RoPE (cos, sin) of the
// lane's four features at that position, and the four features' norm gains.
// Cluster launches load them while the MMAs run (under a full-rate weight
// stream they would miss L2 after it).
struct ColOps {
  int pos[4], strm[4], rend[4];
  float2 cs[4][4];
  float g[4];
};

// tmeta: the chunk's token metadata staged in shared memory
// (stage_token_meta), or nullptr to read it from the epilogue arguments.
// Columns at or past nvalid (or N) get position 0: their values are never
// stored.
__device__ __forceinline__ void col_ops_load(const GemmArgs& a, int m_tile, int n0, int nvalid, int q, int lane,
                                             const int* tmeta, ColOps& o) {
  const int sidx = seg_of_tile(a, m_tile);
  const HeadSeg& sg = a.epi.seg[sidx];
  const int d = a.epi.head_dim;
  const int half = d >> 1;
  const bool rot = sg.kind != HEAD_V;
#pragma unroll
  for (int jj = 0; jj < 4; ++jj) {
    const int j = q + 4 * jj;
    const int t = n0 + j;
    int p = 0, sm = 0, e = 0;
    if (j < nvalid && t < a.N) {
      if (tmeta != nullptr) {
        p = tmeta[4 * j];
        sm = tmeta[4 * j + 1];
        e = tmeta[4 * j + 2];
      } else if (a.epi.pos_mode == 0) {
        sm = a.epi.s_begin + t / 16;
        p = a.epi.lens[sm] + (t & 15);
      } else {
        sm = a.epi.row_stream[t];
        p = a.epi.row_pos[t];
        e = a.epi.row_end[t];
      }
    }
    o.pos[jj] = p;
    o.strm[jj] = sm;
    o.rend[jj] = e;
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int dim = (lane + 32 * i) & (d - 1);  // d divides the tile's 128 rows
    const int fi = dim < half ? dim : dim - half;
    o.g[i] = rot ? __bfloat162float(sg.gain[dim]) : 1.f;
#pragma unroll
    for (int jj = 0; jj < 4; ++jj)
      o.cs[jj][i] = rot ? a.epi.rope[static_cast<int64_t>(o.pos[jj]) * half + fi] : make_float2(1.f, 0.f);
  }
}

// Heads epilogue of a whole tile (row-table mode or block mode): the
// position, stream and segment end of its n tokens go to shared memory once,
// meta[4 * c + {0, 1, 2}], instead of being loaded per chunk by every thread.
__device__ __forceinline__ void stage_token_meta(const GemmArgs& a, int t0, int n, int row, int* meta) {
  named_bar_sync(1, 128);  // the previous tile's chunks are done with meta
  for (int c = row; c < n; c += 128) {
    const int t = t0 + c;
    int p = 0, sm = 0, e = 0;
    if (t < a.N) {
      if (a.epi.pos_mode == 0) {
        sm = a.epi.s_begin + t / 16;
        p = a.epi.lens[sm] + (t & 15);
      } else {
        sm = a.epi.row_stream[t];
        p = a.epi.row_pos[t];
        e = a.epi.row_end[t];
      }
    }
    meta[4 * c] = p;
    meta[4 * c + 1] = sm;
    meta[4 * c + 2] = e;
  }
  named_bar_sync(1, 128);
}

// The residual rows X[n0 .. n0+15][m] a residual epilogue chunk adds to.
__device__ __forceinline__ void resid_load(const GemmArgs& a, int m, int n0, int nvalid, float (&xo)[16]) {
  const float* X = static_cast<const float*>(a.epi.out);
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int t = n0 + j;
    xo[j] = (j < nvalid && t < a.N && m < a.M) ? X[static_cast<int64_t>(t) * a.epi.ldo + m] : 0.f;
  }
}

// xpre (residual epilogue): the chunk's X values, loaded earlier by the
// caller (so a wide tile's next chunk loads while this one computes).
template <int EPI>
__device__ __forceinline__ void epi_chunk(const GemmArgs& a, int m_tile, int n0, int row, int q, int lane,
                                          const float (&v0)[16], const float (&v1)[16], float* xch, float* red,
                                          int nvalid = 16, const float (*xpre)[16] = nullptr) {
  const int m = m_tile * kTileM + row;
  if constexpr (EPI == EPI_RESID) {
    // X += v, and the tile's per-column sums of squares of the new X
    // all 16 loads are issued before the first store: interleaved, a store
    // to X could alias the next load, and the loads would run one at a time
    float ss[16], xo[16];
    float* X = static_cast<float*>(a.epi.out);
    if (xpre != nullptr) {
#pragma unroll
      for (int j = 0; j < 16; ++j) xo[j] = (*xpre)[j];
    } else {
      resid_load(a, m, n0, nvalid, xo);
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int t = n0 + j;
      ss[j] = 0.f;
      if (j < nvalid && t < a.N && m < a.M) {
        const float xn = xo[j] + v0[j];
        X[static_cast<int64_t>(t) * a.epi.ldo + m] = xn;
        ss[j] = xn * xn;
      }
    }
    if (a.epi.ss_out) publish_ss(a, ss, m_tile, n0, row, q, lane, red, nvalid);
  } else if constexpr (EPI == EPI_STORE_F32) {
    // y = v, and (optionally) the tile's per-column sums of squares of y
    float ss[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int t = n0 + j;
      ss[j] = 0.f;
      if (j < nvalid && t < a.N && m < a.M) {
        static_cast<float*>(a.epi.out)[static_cast<int64_t>(t) * a.epi.ldo + m] = v0[j];
        ss[j] = v0[j] * v0[j];
      }
    }
    if (a.epi.ss_out) publish_ss(a, ss, m_tile, n0, row, q, lane, red, nvalid);
  } else if constexpr (EPI == EPI_STORE_BF16) {
    float y[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int t = n0 + j;
      const __nv_bfloat16 b = __float2bfloat16_rn(v0[j]);
      y[j] = __bfloat162float(b);
      if (j < nvalid && t < a.N && m < a.M) static_cast<__nv_bfloat16*>(a.epi.out)[static_cast<int64_t>(t) * a.epi.ldo + m] = b;
    }
    if (a.epi.cand_k > 0) {
      // per column: the tile's top cand_k rows (warp q takes columns q, q + 4,
      // q + 8, q + 12), lane l holding rows l + 32i
#pragma unroll
      for (int j = 0; j < 16; ++j) xch[j * (kTileM + 1) + row] = m < a.M ? y[j] : -INFINITY;
      named_bar_sync(1, 128);
      // the warp's four columns go through the k rounds together, so their
      // shuffle chains overlap (each column's selection is unchanged)
      float lv[4][4];
      uint32_t used[4];
      bool live[4];
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const int j = q + 4 * jj;
        live[jj] = j < nvalid && n0 + j < a.N;
        used[jj] = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) lv[jj][i] = xch[j * (kTileM + 1) + lane + 32 * i];
      }
      for (int r = 0; r < a.epi.cand_k; ++r) {
        float bv[4];
        int bi[4];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          // lane-local best unused (rows ascend with i, so strict > keeps the lower row)
          bv[jj] = -INFINITY;
          bi[jj] = 0x7fffffff;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if (!(used[jj] >> i & 1u) && (lv[jj][i] > bv[jj] || bi[jj] == 0x7fffffff)) {
              bv[jj] = lv[jj][i];
              bi[jj] = lane + 32 * i;
            }
          }
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) {
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv[jj], off);
            const int oi = __shfl_xor_sync(0xffffffffu, bi[jj], off);
            if (ov > bv[jj] || (ov == bv[jj] && oi < bi[jj])) {
              bv[jj] = ov;
              bi[jj] = oi;
            }
          }
        }
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          if (bi[jj] != 0x7fffffff && (bi[jj] & 31) == lane) used[jj] |= 1u << (bi[jj] >> 5);
          if (lane == 0 && live[jj]) {
            const int64_t base = (static_cast<int64_t>(n0 + q + 4 * jj) * a.m_tiles + m_tile) * a.epi.cand_k;
            a.epi.cand_v[base + r] = bv[jj];
            a.epi.cand_i[base + r] = bi[jj] == 0x7fffffff ? 0x7fffffff : m_tile * kTileM + bi[jj];
          }
        }
      }
      named_bar_sync(1, 128);  // xch reusable by the next chunk
    }
  } else if constexpr (EPI == EPI_SWIGLU) {
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int t = n0 + j;
      if (j >= nvalid || t >= a.N) break;
      const int64_t o = static_cast<int64_t>(t) * a.epi.ldo + m;
      static_cast<__nv_bfloat16*>(a.epi.out)[o] = __float2bfloat16_rn(silu_f(v0[j]) * v1[j]);
    }
  }
}

// Heads epilogue (per-head RMSNorm over d with q_norm / k_norm gains,
// rotate-half RoPE, bf16 out) of one chunk of up to 16 columns, a warp per
// column: the chunk's fp32 accumulators pass through shared memory
// (xch[j][129]), then warp w takes columns w, w + 4, w + 8, w + 12 with lane l
// holding the tile's features l + 32 i (i = 0..3), so a head's sum of squares
// and the RoPE partner (feature -+ d/2) are inside one warp: the partner is
// slice i ^ 2 (d = 128), i ^ 1 (d = 64) or lane l ^ 16 (d = 32). Each slice's
// sum is the xor butterfly over offsets 16, 8, 4, 2, 1 and the slices of a
// head add in feature order. Columns at or past nvalid are not stored.
__device__ __forceinline__ void heads_cols(const GemmArgs& a, int m_tile, int n0, int row, int q, int lane,
                                           const float (&v0)[16], float* xch, int nvalid, const ColOps& o) {
  const int sidx = seg_of_tile(a, m_tile);
  const HeadSeg& sg = a.epi.seg[sidx];
  const int d = a.epi.head_dim;
  const int half = d >> 1;
  const int fbase = (m_tile - a.a_seg_tile[sidx]) * kTileM;  // the tile's first feature in the projection
  const bool rot = sg.kind != HEAD_V;
  named_bar_sync(1, 128);  // the previous chunk's columns are done with xch
#pragma unroll
  for (int j = 0; j < 16; ++j) xch[j * (kTileM + 1) + row] = v0[j];
  named_bar_sync(1, 128);
  const float inv_d = 1.0f / static_cast<float>(d);  // d is a power of two: exact
  // the four columns go through each step together (independent chains)
  float y[4][4];
#pragma unroll
  for (int jj = 0; jj < 4; ++jj)
#pragma unroll
    for (int i = 0; i < 4; ++i) y[jj][i] = xch[(q + 4 * jj) * (kTileM + 1) + lane + 32 * i];
  if (rot) {
    float sq[4][4];
#pragma unroll
    for (int jj = 0; jj < 4; ++jj)
#pragma unroll
      for (int i = 0; i < 4; ++i) sq[jj][i] = y[jj][i] * y[jj][i];
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1)
#pragma unroll
      for (int jj = 0; jj < 4; ++jj)
#pragma unroll
        for (int i = 0; i < 4; ++i) sq[jj][i] += __shfl_xor_sync(0xffffffffu, sq[jj][i], off);
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      float hs[4];
      if (d == 128) {
        const float s4 = ((sq[jj][0] + sq[jj][1]) + sq[jj][2]) + sq[jj][3];
        hs[0] = hs[1] = hs[2] = hs[3] = s4;
      } else if (d == 64) {
        hs[0] = hs[1] = sq[jj][0] + sq[jj][1];
        hs[2] = hs[3] = sq[jj][2] + sq[jj][3];
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) hs[i] = sq[jj][i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
        y[jj][i] = head_norm_apply(y[jj][i], head_norm_scale(hs[i], inv_d, a.epi.eps), o.g[i]);
    }
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      float yp[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        yp[i] = d == 128 ? y[jj][i ^ 2] : d == 64 ? y[jj][i ^ 1] : __shfl_xor_sync(0xffffffffu, y[jj][i], 16);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int dim = (lane + 32 * i) & (d - 1);
        y[jj][i] = rope_rotate(y[jj][i], yp[i], o.cs[jj][i], dim < half);
      }
    }
  }
#pragma unroll
  for (int jj = 0; jj < 4; ++jj) {
    const int j = q + 4 * jj;
    const int t = n0 + j;
    if (j >= nvalid || t >= a.N) break;
    if (a.epi.pos_mode == 0) {
      __nv_bfloat16* dst = sg.dst + static_cast<int64_t>(t) * (sg.heads * d) + fbase + lane;
#pragma unroll
      for (int i = 0; i < 4; ++i) dst[32 * i] = __float2bfloat16_rn(y[jj][i]);
    } else {
      // a later row of the same segment owns this ring slot
      const int pos = o.pos[jj];
      if (sg.window > 0 && pos < o.rend[jj] - sg.window) continue;
      const int slot = sg.window > 0 ? (pos % sg.window) : pos;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int f = fbase + lane + 32 * i;
        sg.dst[((static_cast<int64_t>(o.strm[jj]) * sg.heads + f / d) * sg.cap + slot) * d + (f & (d - 1))] =
            __float2bfloat16_rn(y[jj][i]);
      }
    }
  }
}

// ---------------------------------------------------------------- kernel
template <int BN, bool DUAL, int STAGES, int EPI, int MINB, bool CLU>
__global__ void __launch_bounds__(kGemmThreads, MINB) gemm_kernel(const __grid_constant__ GemmArgs args) {
  using Tr = GemmTraits<BN, DUAL, STAGES, EPI>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* tiles = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(tiles + STAGES * Tr::kStageBytes);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + Tr::kAccBufs;
  uint64_t* drain = tempty + Tr::kAccBufs;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_word = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* last_word = abort_word + 1;
  float* xch = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(full) + Tr::kBarBytes);
  float* red = xch + Tr::kXchFloats;
  int* tmeta = reinterpret_cast<int*>(red + Tr::kRedFloats);  // heads: the tile's token metadata

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  int clu_tile = -1;  // cluster split-K: this CTA's unit, once its partial is parked
  ColOps cpre;        // heads epilogue operands, preloaded (cluster launches)
  float xpre[16];     // residual epilogue: this rank's X values, preloaded (cluster launches)
  bool have_pre = false;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < Tr::kAccBufs; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 128);
    }
    mbar_init(drain, 1);
    *abort_word = 0;
    *last_word = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, Tr::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_trigger();

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      for (int i = 0; i < args.n_aseg; ++i) tma_prefetch_desc(&args.a_map[i]);
      const uint64_t pol_w = policy_evict_first();  // weights stream through once
      const uint64_t pol_x = policy_evict_last();   // activations are re-read by every tile
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      bool ok = true;
      bool first = true;
      for (int u = blockIdx.x; u < args.units && ok; u += gridDim.x) {
        int m_tile, kc, n_tile;
        decode_unit<CLU>(args, u, m_tile, kc, n_tile);
        const int kb0 = static_cast<int>(static_cast<long long>(kc) * args.kb_total / args.ksplit);
        const int kb1 = static_cast<int>(static_cast<long long>(kc + 1) * args.kb_total / args.ksplit);
        const int sidx = seg_of_tile(args, m_tile);
        const int arow = (m_tile - args.a_seg_tile[sidx]) * kTileM;
        int kb = kb0;
        if (first) {
          // Weights do not depend on the previous kernel: fill every stage
          // with its weight tile before waiting for the activations.
          first = false;
          const int npre = kb1 - kb0 < STAGES ? kb1 - kb0 : STAGES;
          for (int i = 0; i < npre; ++i) {
            uint8_t* st = tiles + i * Tr::kStageBytes;
            mbar_arrive_expect_tx(&full[i], Tr::kStageBytes);
            tma_load_2d(st, &args.a_map[sidx], &full[i], (kb0 + i) * kTileK, arow, pol_w);
            if constexpr (DUAL) tma_load_2d(st + Tr::kABytes, &args.a2_map, &full[i], (kb0 + i) * kTileK, arow, pol_w);
          }
          pdl_wait();
          for (int i = 0; i < npre; ++i) {
            const int kbi = kb0 + i;
            const int pl = kbi / args.b_plane_kb;
            const int kin = kbi - pl * args.b_plane_kb;
            tma_load_2d(tiles + i * Tr::kStageBytes + Tr::kABytes * (DUAL ? 2 : 1), &args.b_map[pl], &full[i],
                        kin * kTileK, n_tile * BN, pol_x);
          }
          issued = npre;
          kb = kb0 + npre;
          stage = npre % STAGES;
          phase = npre == STAGES ? 1u : 0u;
        }
        for (; kb < kb1; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, args.err, DFLASH_STATUS_TIMEOUT, abort_word)) {
            ok = false;
            break;
          }
          uint8_t* st = tiles + stage * Tr::kStageBytes;
          mbar_arrive_expect_tx(&full[stage], Tr::kStageBytes);
          tma_load_2d(st, &args.a_map[sidx], &full[stage], kb * kTileK, arow, pol_w);
          if constexpr (DUAL) tma_load_2d(st + Tr::kABytes, &args.a2_map, &full[stage], kb * kTileK, arow, pol_w);
          const int pl = kb / args.b_plane_kb;
          const int kin = kb - pl * args.b_plane_kb;
          tma_load_2d(st + Tr::kABytes * (DUAL ? 2 : 1), &args.b_map[pl], &full[stage], kin * kTileK, n_tile * BN,
                      pol_x);
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // make sure no copy is still landing in shared memory when the CTA ends
      for (int s = 0; s < STAGES; ++s) {
        if (issued > s) {
          const uint32_t par = (s < stage) ? phase : (phase ^ 1u);
          mbar_wait(&full[s], par, args.err, DFLASH_STATUS_TIMEOUT, nullptr);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      bool any = false;
      for (int u = blockIdx.x; u < args.units && ok; u += gridDim.x) {
        int m_tile, kc, n_tile;
        decode_unit<CLU>(args, u, m_tile, kc, n_tile);
        const int kb0 = static_cast<int>(static_cast<long long>(kc) * args.kb_total / args.ksplit);
        const int kb1 = static_cast<int>(static_cast<long long>(kc + 1) * args.kb_total / args.ksplit);
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, args.err, DFLASH_STATUS_TIMEOUT, abort_word)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * Tr::kAccCols);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&full[stage], phase, args.err, DFLASH_STATUS_TIMEOUT, abort_word)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(tiles + stage * Tr::kStageBytes);
          const uint32_t b_addr = a_addr + Tr::kABytes * (DUAL ? 2 : 1);
#pragma unroll
          for (int kk = 0; kk < kTileK / 16; ++kk) {
            const uint32_t accum = (kb > kb0 || kk > 0) ? 1u : 0u;
            const uint64_t bdesc = sdesc_sw128(b_addr + kk * 32);
            umma_bf16(d_tmem, sdesc_sw128(a_addr + kk * 32), bdesc, Tr::kIdesc, accum);
            if constexpr (DUAL)
              umma_bf16(d_tmem + BN, sdesc_sw128(a_addr + Tr::kABytes + kk * 32), bdesc, Tr::kIdesc, accum);
          }
          any = true;
          umma_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(&tfull[acc]);
        if (++acc == Tr::kAccBufs) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // all MMAs of this CTA complete before tensor memory is released
      if (any) {
        umma_commit(drain);
        mbar_wait(drain, 0, args.err, DFLASH_STATUS_TIMEOUT, nullptr);
      }
    }
  } else {
    // ------------------------------------------------ epilogue (warps 2..5)
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    const int row = q * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    const bool epi_leader = (warp == 2 && lane == 0);
    pdl_wait();  // the epilogue reads and writes buffers of earlier kernels
    for (int u = blockIdx.x; u < args.units; u += gridDim.x) {
      int m_tile, kc, n_tile;
      decode_unit<CLU>(args, u, m_tile, kc, n_tile);
      if constexpr (EPI == EPI_HEADS && CLU) {
        // the epilogue's gains, positions and RoPE values, loaded while the
        // MMAs run (under a full-rate weight stream they miss L2)
        const int ks = args.ksplit;
        const int rk = static_cast<int>(gemm_cluster_rank());
        const int cb = rk * BN / ks, ce = (rk + 1) * BN / ks;
        if (ce - cb <= 16) {
          col_ops_load(args, m_tile, n_tile * BN + cb, ce - cb, q, lane, nullptr, cpre);
          have_pre = true;
        }
      } else if constexpr (EPI == EPI_RESID && CLU) {
        // the residual this rank adds to (final: the epilogue is past its PDL wait)
        const int ks = args.ksplit;
        const int rk = static_cast<int>(gemm_cluster_rank());
        const int cb = rk * BN / ks, ce = (rk + 1) * BN / ks;
        if (ce - cb <= 16) {
          resid_load(args, m_tile * kTileM + row, n_tile * BN + cb, ce - cb, xpre);
          have_pre = true;
        }
      } else if constexpr (EPI == EPI_HEADS) {
        // the epilogue's per-head gain and RoPE rows are read once, long after
        // the weight stream has evicted them: pull them into L2 now
        if (args.epi.pos_mode == 0) {
          const int sidx = seg_of_tile(args, m_tile);
          const HeadSeg& sg = args.epi.seg[sidx];
          const int half = args.epi.head_dim >> 1;
          const int lpr = (half * 8 + 127) / 128;  // 128-byte lines per RoPE row
          for (int i = row; i < BN * lpr; i += 128) {
            const int t = n_tile * BN + i / lpr;
            if (t < args.N) {
              const int p = args.epi.lens[args.epi.s_begin + t / 16] + (t & 15);
              prefetch_l2(reinterpret_cast<const char*>(args.epi.rope + static_cast<int64_t>(p) * half) +
                          (i % lpr) * 128);
            }
          }
          if (sg.gain != nullptr && row * 64 < args.epi.head_dim) prefetch_l2(sg.gain + row * 64);
        }
      }
      const bool ok = mbar_wait(&tfull[acc], acc_phase, args.err, DFLASH_STATUS_TIMEOUT, abort_word);
      // the four epilogue warps leave together, so none is left at a named barrier
      if (named_bar_or(1, 128, ok ? 0 : 1)) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * Tr::kAccCols);
      float v0[16], v1[16];
      if constexpr (CLU) {
        // park this chunk's fp32 partial in the idle stage memory, [acc][col][row]
        float* part = reinterpret_cast<float*>(tiles);
        for (int c0 = 0; c0 < BN; c0 += 16) {
          tmem_ld16(tbase + c0, v0);
#pragma unroll
          for (int j = 0; j < 16; ++j) part[(c0 + j) * kTileM + row] = v0[j];
          if constexpr (DUAL) {
            tmem_ld16(tbase + BN + c0, v1);
#pragma unroll
            for (int j = 0; j < 16; ++j) part[(BN + c0 + j) * kTileM + row] = v1[j];
          }
        }
        tc_fence_before();
        mbar_arrive(&tempty[acc]);
        clu_tile = u;  // reduced after the cluster barrier below
      } else if (args.ksplit == 1) {
        if constexpr (EPI == EPI_HEADS) stage_token_meta(args, n_tile * BN, BN, row, tmeta);
        const int m = m_tile * kTileM + row;
        float xn[16];  // residual: the next chunk's X, loaded a chunk ahead
        if constexpr (EPI == EPI_RESID) resid_load(args, m, n_tile * BN, 16, xn);
        for (int c0 = 0; c0 < BN; c0 += 16) {
          tmem_ld16(tbase + c0, v0);
          if constexpr (DUAL) tmem_ld16(tbase + BN + c0, v1);
          if constexpr (EPI == EPI_HEADS) {
            ColOps o;
            col_ops_load(args, m_tile, n_tile * BN + c0, 16, q, lane, tmeta + 4 * c0, o);
            heads_cols(args, m_tile, n_tile * BN + c0, row, q, lane, v0, xch, 16, o);
          } else if constexpr (EPI == EPI_RESID) {
            float xc[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) xc[j] = xn[j];
            if (c0 + 16 < BN) resid_load(args, m, n_tile * BN + c0 + 16, 16, xn);
            epi_chunk<EPI>(args, m_tile, n_tile * BN + c0, row, q, lane, v0, v1, xch, red, 16, &xc);
          } else {
            epi_chunk<EPI>(args, m_tile, n_tile * BN + c0, row, q, lane, v0, v1, xch, red);
          }
        }
        tc_fence_before();
        mbar_arrive(&tempty[acc]);
      } else {
        float* slot = args.partial + static_cast<size_t>(u) * (Tr::kAcc * BN * kTileM);
        for (int c0 = 0; c0 < BN; c0 += 16) {
          tmem_ld16(tbase + c0, v0);
#pragma unroll
          for (int j = 0; j < 16; ++j) slot[(c0 + j) * kTileM + row] = v0[j];
          if constexpr (DUAL) {
            tmem_ld16(tbase + BN + c0, v1);
#pragma unroll
            for (int j = 0; j < 16; ++j) slot[(BN + c0 + j) * kTileM + row] = v1[j];
          }
        }
        tc_fence_before();
        mbar_arrive(&tempty[acc]);
        __threadfence();
        named_bar_sync(1, 128);
        if (epi_leader) {
          const int old = atomicAdd(&args.counters[(m_tile - args.m_tile0) * args.n_tiles + n_tile], 1);
          *last_word = (old == args.ksplit - 1) ? 1 : 0;
        }
        named_bar_sync(1, 128);
        const bool last = *last_word != 0;
        if (last) {
          __threadfence();
          if constexpr (EPI == EPI_HEADS) stage_token_meta(args, n_tile * BN, BN, row, tmeta);
          const int m = m_tile * kTileM + row;
          float xn[16];  // residual: the next chunk's X, loaded a chunk ahead
          if constexpr (EPI == EPI_RESID) resid_load(args, m, n_tile * BN, 16, xn);
          for (int c0 = 0; c0 < BN; c0 += 16) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              v0[j] = 0.f;
              v1[j] = 0.f;
            }
            // chunk order; the loads of two chunks are issued before their adds
            for (int k2 = 0; k2 < args.ksplit; k2 += 2) {
              const bool two = k2 + 1 < args.ksplit;
              const float* sa =
                  args.partial + static_cast<size_t>(((m_tile - args.m_tile0) * args.ksplit + k2) * args.n_tiles + n_tile) *
                                     (Tr::kAcc * BN * kTileM);
              const float* sb = two ? sa + static_cast<size_t>(args.n_tiles) * (Tr::kAcc * BN * kTileM) : sa;
              float a0[16], b0[16], a1[16], b1[16];
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                a0[j] = __ldcg(&sa[(c0 + j) * kTileM + row]);
                b0[j] = two ? __ldcg(&sb[(c0 + j) * kTileM + row]) : 0.f;
                if constexpr (DUAL) {
                  a1[j] = __ldcg(&sa[(BN + c0 + j) * kTileM + row]);
                  b1[j] = two ? __ldcg(&sb[(BN + c0 + j) * kTileM + row]) : 0.f;
                }
              }
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                v0[j] += a0[j];
                if (two) v0[j] += b0[j];
                if constexpr (DUAL) {
                  v1[j] += a1[j];
                  if (two) v1[j] += b1[j];
                }
              }
            }
            if constexpr (EPI == EPI_HEADS) {
              ColOps o;
              col_ops_load(args, m_tile, n_tile * BN + c0, 16, q, lane, tmeta + 4 * c0, o);
              heads_cols(args, m_tile, n_tile * BN + c0, row, q, lane, v0, xch, 16, o);
            } else if constexpr (EPI == EPI_RESID) {
              float xc[16];
#pragma unroll
              for (int j = 0; j < 16; ++j) xc[j] = xn[j];
              if (c0 + 16 < BN) resid_load(args, m, n_tile * BN + c0 + 16, 16, xn);
              epi_chunk<EPI>(args, m_tile, n_tile * BN + c0, row, q, lane, v0, v1, xch, red, 16, &xc);
            } else {
              epi_chunk<EPI>(args, m_tile, n_tile * BN + c0, row, q, lane, v0, v1, xch, red);
            }
          }
        }
      }
      if (++acc == Tr::kAccBufs) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  if constexpr (CLU) {
    // every chunk's partial is parked: rank r reduces columns
    // [r*BN/ks, (r+1)*BN/ks) over the cluster, in rank order, and runs the
    // epilogue on them; the second barrier keeps the partials alive until
    // every rank has read them
    __syncwarp();
    gemm_cluster_sync();
    bool arrived = false;
    if (warp >= 2 && named_bar_or(1, 128, clu_tile < 0 ? 1 : 0) == 0) {
      int m_tile, kc, n_tile;
      decode_unit<CLU>(args, clu_tile, m_tile, kc, n_tile);
      const int q = warp & 3;
      const int row = q * 32 + lane;
      const int ks = args.ksplit;
      const int rk = static_cast<int>(gemm_cluster_rank());
      const int cb = rk * BN / ks, ce = (rk + 1) * BN / ks;
      const uint32_t pbase = smem_u32(tiles);
      float v0[16], v1[16];
      for (int c0 = cb; c0 < ce; c0 += 16) {
        const int nv = ce - c0 < 16 ? ce - c0 : 16;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          v0[j] = 0.f;
          v1[j] = 0.f;
        }
        if (!DUAL && nv <= 4) {
          // few columns a rank (batch-1 tiles): several ranks' loads in flight
          // at once (four beside the heads epilogue's preloaded operands)
          constexpr int kR = EPI == EPI_HEADS ? 4 : kMaxClusterSplit;
          for (int r0 = 0; r0 < ks; r0 += kR) {
            float buf[kR][4];
#pragma unroll
            for (int r = 0; r < kR; ++r) {
              const uint32_t ra = gemm_mapa(pbase, static_cast<uint32_t>(r0 + r < ks ? r0 + r : r0));
#pragma unroll
              for (int j = 0; j < 4; ++j)
                buf[r][j] = (r0 + r < ks && j < nv)
                                ? gemm_ld_dsmem(ra + static_cast<uint32_t>(((c0 + j) * kTileM + row) * 4))
                                : 0.f;
            }
#pragma unroll
            for (int r = 0; r < kR; ++r) {
              if (r0 + r < ks) {
#pragma unroll
                for (int j = 0; j < 4; ++j) v0[j] += buf[r][j];
              }
            }
          }
        } else {
          // rank order; the loads of two ranks are issued before their adds
          for (int r2 = 0; r2 < ks; r2 += 2) {
            const bool two = r2 + 1 < ks;
            const uint32_t ra = gemm_mapa(pbase, static_cast<uint32_t>(r2));
            const uint32_t rb = gemm_mapa(pbase, static_cast<uint32_t>(two ? r2 + 1 : r2));
            float a0[16], b0[16], a1[16], b1[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const uint32_t o0 = static_cast<uint32_t>(((c0 + j) * kTileM + row) * 4);
              const uint32_t o1 = static_cast<uint32_t>(((BN + c0 + j) * kTileM + row) * 4);
              a0[j] = j < nv ? gemm_ld_dsmem(ra + o0) : 0.f;
              b0[j] = (j < nv && two) ? gemm_ld_dsmem(rb + o0) : 0.f;
              if constexpr (DUAL) {
                a1[j] = j < nv ? gemm_ld_dsmem(ra + o1) : 0.f;
                b1[j] = (j < nv && two) ? gemm_ld_dsmem(rb + o1) : 0.f;
              }
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              v0[j] += a0[j];
              if (two) v0[j] += b0[j];
              if constexpr (DUAL) {
                v1[j] += a1[j];
                if (two) v1[j] += b1[j];
              }
            }
          }
        }
        if (c0 + 16 >= ce) {
          // the last remote reads are in registers: the other ranks may go
          gemm_cluster_arrive();
          arrived = true;
        }
        if constexpr (EPI == EPI_HEADS) {
          if (have_pre) {
            heads_cols(args, m_tile, n_tile * BN + c0, row, q, lane, v0, xch, nv, cpre);
          } else {
            ColOps o;
            col_ops_load(args, m_tile, n_tile * BN + c0, nv, q, lane, nullptr, o);
            heads_cols(args, m_tile, n_tile * BN + c0, row, q, lane, v0, xch, nv, o);
          }
        } else if constexpr (EPI == EPI_RESID) {
          epi_chunk<EPI>(args, m_tile, n_tile * BN + c0, row, q, lane, v0, v1, xch, red, nv,
                         have_pre ? &xpre : nullptr);
        } else {
          epi_chunk<EPI>(args, m_tile, n_tile * BN + c0, row, q, lane, v0, v1, xch, red, nv);
        }
      }
    }
    if (!arrived) gemm_cluster_arrive();
    gemm_cluster_wait();  // the partials stay alive until every rank has read them
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, Tr::kTmemCols);
}

// ---------------------------------------------------------------- host side
namespace {

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn get_encode() {
  static EncodeFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(p);
  }
  return fn;
}

template <int BN, bool DUAL, int STAGES, int EPI, int MINB, bool CLU>
int launch_inst(const GemmArgs& a, int num_sms, cudaStream_t st) {
  using Tr = GemmTraits<BN, DUAL, STAGES, EPI>;
  auto kern = gemm_kernel<BN, DUAL, STAGES, EPI, MINB, CLU>;
  static bool configured = false;
  if (!configured) {
    // two CTAs of the batch-1 variants share an SM only with the full carveout
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Tr::kSmemBytes) != cudaSuccess ||
        cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess)
      return DFLASH_E_CUDA;
    configured = true;
  }
  cudaError_t e;
  if constexpr (CLU) {
    // one unit per CTA, the ksplit chunks of a tile form one cluster
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(a.ksplit);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(a.units);
    cfg.blockDim = dim3(kGemmThreads);
    cfg.dynamicSmemBytes = Tr::kSmemBytes;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, kern, a);
  } else {
    const int grid = std::max(1, std::min(a.units, num_sms * MINB));
    e = launch_pdl(kern, dim3(grid), dim3(kGemmThreads), Tr::kSmemBytes, st, a);
  }
  count_launch();
  return cuda_status(e);
}

template <int BN, bool DUAL, int STAGES, int MINB, int EPI>
int launch_mode(const GemmArgs& a, int num_sms, cudaStream_t st) {
  using Tr = GemmTraits<BN, DUAL, STAGES, EPI>;
  if (a.ksplit > 1 && a.ksplit <= kMaxClusterSplit && !a.no_cluster) {
    if constexpr (Tr::kClusterFits) return launch_inst<BN, DUAL, STAGES, EPI, MINB, true>(a, num_sms, st);
  }
  return launch_inst<BN, DUAL, STAGES, EPI, MINB, false>(a, num_sms, st);
}

template <int BN, bool DUAL, int STAGES, int MINB>
int launch_epi(const GemmArgs& a, int epi, int num_sms, cudaStream_t st) {
  switch (epi) {
    case EPI_STORE_F32:
      if constexpr (!DUAL) return launch_mode<BN, DUAL, STAGES, MINB, EPI_STORE_F32>(a, num_sms, st);
      break;
    case EPI_STORE_BF16:
      if constexpr (!DUAL) return launch_mode<BN, DUAL, STAGES, MINB, EPI_STORE_BF16>(a, num_sms, st);
      break;
    case EPI_RESID:
      if constexpr (!DUAL) return launch_mode<BN, DUAL, STAGES, MINB, EPI_RESID>(a, num_sms, st);
      break;
    case EPI_HEADS:
      if constexpr (!DUAL) return launch_mode<BN, DUAL, STAGES, MINB, EPI_HEADS>(a, num_sms, st);
      break;
    case EPI_SWIGLU:
      if constexpr (DUAL) return launch_mode<BN, DUAL, STAGES, MINB, EPI_SWIGLU>(a, num_sms, st);
      break;
    default:
      break;
  }
  return DFLASH_E_INVALID_ARG;
}

}  // namespace

int encode_kmajor_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int64_t ld, int box_rows) {
  EncodeFn enc = get_encode();
  if (!enc) return DFLASH_E_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(base) & 15u) != 0 || (ld * 2) % 16 != 0 || cols % kTileK != 0)
    return DFLASH_E_SHAPE;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld * 2)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kTileK), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DFLASH_OK : DFLASH_E_CUDA;
}

int gemm_bn_for(int N) {
  if (N <= 16) return 16;
  if (N <= 128) return 128;
  return 256;
}

int gemm_choose_ksplit(int m_tiles, int kb_total, int num_sms) {
  // The largest split (<= kMaxClusterSplit, >= 4 reduction blocks a chunk)
  // whose CTAs all fit in one wave of clusters at two CTAs an SM. Cluster
  // placement inside GPCs leaves some SMs unused, so the wave is taken as
  // 85% of 2 x SMs (measured on GB300: 48 tiles x 5 splits runs in one wave,
  // x 6 in two).
  const int budget = (2 * num_sms * 85) / 100;
  int best = 1;
  for (int ks = 2; ks <= kMaxClusterSplit; ++ks) {
    if (kb_total / ks < 4) break;
    if (m_tiles * ks <= budget) best = ks;
  }
  return best;
}

static void fill_args(const GemmPlan& p, GemmArgs& a, int BN) {
  a.n_aseg = p.n_aseg;
  a.a_seg_tile[0] = 0;
  for (int i = 0; i < p.n_aseg; ++i) {
    a.a_map[i] = *p.a_maps[i];
    a.a_seg_tile[i + 1] = a.a_seg_tile[i] + p.a_rows[i] / kTileM;
  }
  if (p.a2_map) a.a2_map = *p.a2_map;
  a.m_tile0 = p.m_tile0;
  a.M = p.m_tile0 * kTileM + p.M;  // the end row: epilogue row indices are the weight's
  a.N = p.N;
  a.K = p.K;
  a.m_tiles = p.M / kTileM;
  a.n_tiles = (p.N + BN - 1) / BN;
  a.kb_total = p.K / kTileK;
  a.b_plane_kb = p.Kp / kTileK;
  a.ksplit = p.ksplit;
  a.units = a.m_tiles * a.n_tiles * a.ksplit;
  a.no_cluster = p.no_cluster;
  a.epi = p.epi_args;
}

size_t gemm_partial_bytes(const GemmPlan& p) {
  if (p.ksplit <= 1) return 0;
  const int BN = plan_bn(p);
  const size_t units = static_cast<size_t>(p.M / kTileM) * ((p.N + BN - 1) / BN) * p.ksplit;
  return units * (p.a2_map ? 2 : 1) * BN * kTileM * sizeof(float);
}

size_t gemm_counter_count(const GemmPlan& p) {
  const int BN = plan_bn(p);
  return static_cast<size_t>(p.M / kTileM) * ((p.N + BN - 1) / BN);
}

int gemm_launch(const GemmPlan& p, float* partial, int* counters, int* err, int num_sms, cudaStream_t st) {
  if (p.M % kTileM || p.K % kTileK || p.Kp % kTileK || p.N <= 0 || p.n_aseg < 1 || p.n_aseg > kMaxASeg ||
      p.n_b < 1 || p.n_b > kMaxBPlane || p.Kp * p.n_b != p.K || (p.bn != 0 && p.bn != 16 && p.bn != 128 && p.bn != 256))
    return DFLASH_E_SHAPE;
  const int BN = plan_bn(p);
  static thread_local GemmArgs a;  // ~4 KiB: kept off the stack
  memset(&a, 0, sizeof(a));
  fill_args(p, a, BN);
  for (int i = 0; i < p.n_b; ++i) {
    const int rc = encode_kmajor_map(&a.b_map[i], p.b_ptr[i], p.N, p.Kp, p.ldb, BN);
    if (rc) return rc;
  }
  a.partial = partial;
  a.counters = counters;
  a.err = err;
  if (a.ksplit > 1 && (partial == nullptr || counters == nullptr)) return DFLASH_E_WORKSPACE;
  const bool dual = p.a2_map != nullptr;
  // algorithmic traffic: weights once, activations once, outputs once
  // (a residual add reads and writes its fp32 row)
  const double M = p.M, N = p.N, K = p.K;
  double out_b = 2.0;
  if (p.epi == EPI_STORE_F32) out_b = 4.0;
  if (p.epi == EPI_RESID) out_b = 8.0;
  const double bytes = (dual ? 2.0 : 1.0) * M * K * 2.0 + N * K * 2.0 + N * M * out_b;
  const double flops = (dual ? 2.0 : 1.0) * 2.0 * M * N * K;
  TraceScope ts(st, p.name, bytes, flops);
  if (BN == 16) {
    return dual ? launch_epi<16, true, 3, 2>(a, p.epi, num_sms, st) : launch_epi<16, false, 5, 2>(a, p.epi, num_sms, st);
  } else if (BN == 128) {
    return dual ? launch_epi<128, true, 4, 1>(a, p.epi, num_sms, st)
                : launch_epi<128, false, 6, 1>(a, p.epi, num_sms, st);
  }
  return dual ? launch_epi<256, true, 3, 1>(a, p.epi, num_sms, st) : launch_epi<256, false, 4, 1>(a, p.epi, num_sms, st);
}

}  // namespace dfl
