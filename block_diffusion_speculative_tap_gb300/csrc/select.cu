// Vocabulary-wide selection: per-row top-k (ties to the lower id), argmax,
// inverse-CDF sampling from softmax(logits / T), and target verification
// (greedy longest-prefix + bonus; speculative sampling with the residual
// max(p - q, 0)).
//
// A row is scanned by one CTA of 16 warps. Warp w owns a contiguous slice of
// the row and reads it 8 bf16 (16 bytes) per lane per step, lanes interleaved,
// so loads are coalesced and every warp's elements are visited in ascending
// id order. Cumulative sums for inverse-CDF draws follow that fixed order
// (per-lane 8-element sums, a warp scan, then the warps in order), so a draw
// is deterministic.
#include <float.h>

#include "internal.h"
#include "ptx.cuh"

namespace dfl {

namespace {

constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kKMax = DFLASH_MAX_TOPK;

struct Slice {
  int g0, g1;  // 8-element groups [g0, g1) owned by this warp
};

__device__ __forceinline__ Slice warp_slice(int V, int w) {
  const int ng = V >> 3;
  return {static_cast<int>(static_cast<long long>(ng) * w / kSelWarps),
          static_cast<int>(static_cast<long long>(ng) * (w + 1) / kSelWarps)};
}

__device__ __forceinline__ void load8(const __nv_bfloat16* row, int g, float (&x)[8]) {
  const uint4 raw = *reinterpret_cast<const uint4*>(row + static_cast<int64_t>(g) * 8);
  const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(p[i]);
    x[2 * i] = f.x;
    x[2 * i + 1] = f.y;
  }
}

// The 8 bf16 values of a 16-byte piece as floats.
__device__ __forceinline__ void unpack8(const uint4& raw, float (&x)[8]) {
  const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(p[i]);
    x[2 * i] = f.x;
    x[2 * i + 1] = f.y;
  }
}

// The largest of the 8 bf16 values of a 16-byte piece, as a float: packed
// bf16 maxima (exact, no rounding), then one conversion a half.
__device__ __forceinline__ float max8(const uint4& raw) {
  const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&raw);
  const __nv_bfloat162 m = __hmax2(__hmax2(p[0], p[1]), __hmax2(p[2], p[3]));
  return fmaxf(__low2float(m), __high2float(m));
}

// (va, ia) ranks before (vb, ib): larger value, then lower id
__device__ __forceinline__ bool better(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

// Inserts (x, xi) into a thread's sorted list (larger value, then lower id).
template <int KM>
__device__ __forceinline__ void list_insert(float (&v)[KM], int (&id)[KM], float x, int xi) {
  if (!better(x, xi, v[KM - 1], id[KM - 1])) return;
  v[KM - 1] = x;
  id[KM - 1] = xi;
#pragma unroll
  for (int j = KM - 1; j > 0; --j) {
    if (better(v[j], id[j], v[j - 1], id[j - 1])) {
      const float tv = v[j];
      v[j] = v[j - 1];
      v[j - 1] = tv;
      const int ti = id[j];
      id[j] = id[j - 1];
      id[j - 1] = ti;
    }
  }
}

// The best of every lane's (v, i) over the warp; all lanes receive it.
__device__ __forceinline__ void warp_best(float& v, int& i) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, off);
    const int oi = __shfl_xor_sync(0xffffffffu, i, off);
    if (better(ov, oi, v, i)) {
      v = ov;
      i = oi;
    }
  }
}

// Block top-k (k <= KM) from every thread's sorted list, by warp shuffles:
// each warp takes its own best k in k rounds (the winner pops its head), the
// 16 warp lists meet in shared memory, and warp 0 merges them in k rounds
// (lane w walks warp w's list). Thread 0 writes ids / vals[r] for r < k; the
// block maximum is returned to every thread.
template <int KM>
__device__ float block_topk(float (&v)[KM], int (&id)[KM], int k, int* ids, float* vals, float* wv, int* wi) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int r = 0; r < k; ++r) {
    float bv = v[0];
    int bi = id[0];
    warp_best(bv, bi);
    if (id[0] == bi) {
#pragma unroll
      for (int j = 0; j < KM - 1; ++j) {
        v[j] = v[j + 1];
        id[j] = id[j + 1];
      }
      v[KM - 1] = -INFINITY;
      id[KM - 1] = INT_MAX;
    }
    if (lane == 0) {
      wv[w * KM + r] = bv;
      wi[w * KM + r] = bi;
    }
  }
  __syncthreads();
  __shared__ float smx;
  if (w == 0) {
    int pos = 0;
    for (int r = 0; r < k; ++r) {
      float bv = lane < kSelWarps && pos < k ? wv[lane * KM + pos] : -INFINITY;
      int bi = lane < kSelWarps && pos < k ? wi[lane * KM + pos] : INT_MAX;
      const int mine = bi;
      warp_best(bv, bi);
      if (r == 0 && lane == 0) smx = bv;
      if (mine == bi && lane < kSelWarps) ++pos;
      if (lane == 0) {
        ids[r] = bi;
        if (vals) vals[r] = bv;
      }
    }
  }
  __syncthreads();
  return smx;
}

// A warp's running top KM (KM <= 32) of (value, id) pairs, sorted (larger
// value, then lower id): lane j < KM holds the j-th best. A candidate enters
// at the rank counted by a ballot of the better entries, and the entries
// after it move down one lane.
template <int KM>
struct WarpTop {
  float v = -INFINITY;
  int i = INT_MAX;
  __device__ __forceinline__ void insert(float x, int xi, int lane) {
    const unsigned m = __ballot_sync(0xffffffffu, lane < KM && better(v, i, x, xi));
    const int pos = __popc(m);  // the better entries are a prefix
    if (pos >= KM) return;      // warp-uniform
    const float pv = __shfl_up_sync(0xffffffffu, v, 1);
    const int pi = __shfl_up_sync(0xffffffffu, i, 1);
    if (lane > pos && lane < KM) {
      v = pv;
      i = pi;
    }
    if (lane == pos) {
      v = x;
      i = xi;
    }
  }
};

// Top-k (k <= KM <= 16) of the 8-element groups [g_begin, g_end) of a row
// into (ids, vals) (thread 0 writes them); returns the range maximum to every
// thread. The 16 warps split the range into contiguous pieces, lanes
// interleave inside; each warp keeps its exact running top KM across its
// lanes, and a lane's value competes only when it beats the warp's current
// KM-th entry, so after the first few hundred values almost no value leaves
// the load-compare path. Warp 0 merges the 16 warp lists (lane w walks warp
// w's list).
template <int KM>
__device__ float range_topk(const __nv_bfloat16* row, int g_begin, int g_end, int k, int* ids, float* vals) {
  static_assert(KM >= 1 && KM <= 16, "warp lists hold at most 16 entries");
  const int w = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int ng = g_end - g_begin;
  const int wg0 = g_begin + static_cast<int>(static_cast<long long>(ng) * w / kSelWarps);
  const int wg1 = g_begin + static_cast<int>(static_cast<long long>(ng) * (w + 1) / kSelWarps);
  WarpTop<KM> wt;
  float fv = -INFINITY;  // the warp's KM-th entry (lane KM - 1), broadcast
  int fi = INT_MAX;
  float lv = -INFINITY;  // KM == 1: the lane's own running best
  int li = INT_MAX;
  // four 16-byte loads in flight before any is ranked; the trip count is
  // the warp's (every lane reaches the ballots). A piece's largest value
  // is taken on the packed bf16 values; a piece is converted to floats only
  // when it can change the result.
  for (int base = wg0; base < wg1; base += 4 * 32) {
    const int g0 = base + lane;
    uint4 raw[4];
    float gm[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int g = g0 + u * 32;
      raw[u] = g < wg1 ? *reinterpret_cast<const uint4*>(row + static_cast<int64_t>(g) * 8)
                       : make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);  // bf16 -inf
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) gm[u] = max8(raw[u]);
    if constexpr (KM == 1) {
      // arg-max, one warp reduction at the end: a lane's groups arrive in
      // ascending id order, so a group replaces the lane's best only with a
      // strictly larger maximum, taken at its first (lowest) position; an
      // empty lane (li == INT_MAX) also takes a group that only ties
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (g0 + u * 32 < wg1 && (gm[u] > lv || (gm[u] == lv && li == INT_MAX))) {
          float x[8];
          unpack8(raw[u], x);
          int first = 7;
#pragma unroll
          for (int e = 6; e >= 0; --e)
            if (x[e] == gm[u]) first = e;
          lv = gm[u];
          li = (g0 + u * 32) * 8 + first;
        }
      }
    } else {
      if (base == wg0) {
        // The first chunk seeds the floor: t = the KM-th largest of the 32
        // lanes' chunk maxima. At least KM values of this warp's range are
        // >= t, so no value below t can be in its top KM, and the floor
        // (t, worst id) admits exactly the values >= t. Without it every
        // value of the first chunk would take the serial insert path.
        float m = fmaxf(fmaxf(gm[0], gm[1]), fmaxf(gm[2], gm[3]));
        int rank = 0;  // lanes with a larger maximum, ties to the lower lane: a permutation
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float mj = __shfl_sync(0xffffffffu, m, j);
          rank += (mj > m || (mj == m && j < lane)) ? 1 : 0;
        }
        const unsigned who = __ballot_sync(0xffffffffu, rank == KM - 1);
        const float t = __shfl_sync(0xffffffffu, m, __ffs(who) - 1);
        fv = t;
        fi = INT_MAX;
      }
      // a group of 8 whose largest value is below the floor holds no
      // candidate (ties at the floor go on to the exact test); one vote for
      // the whole chunk, since past the first chunks almost none has one
      bool hit = false;
#pragma unroll
      for (int u = 0; u < 4; ++u) hit |= g0 + u * 32 < wg1 && !(gm[u] < fv);
      if (!__any_sync(0xffffffffu, hit)) continue;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (__ballot_sync(0xffffffffu, g0 + u * 32 < wg1 && !(gm[u] < fv)) == 0u) continue;
        float x[8];
        unpack8(raw[u], x);
        // each lane's candidates of this group as an 8-bit mask; one ballot
        // finds the lanes that have any, and only real candidates travel
        const int gid = (g0 + u * 32) * 8;
        uint32_t lm = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e)
          if (g0 + u * 32 < wg1 && better(x[e], gid + e, fv, fi)) lm |= 1u << e;
        unsigned lanes = __ballot_sync(0xffffffffu, lm != 0u);
        while (lanes) {
          const int src = __ffs(lanes) - 1;
          lanes &= lanes - 1;
          uint32_t sm = __shfl_sync(0xffffffffu, lm, src);
          const int sg = __shfl_sync(0xffffffffu, gid, src);
          while (sm) {
            const int e = __ffs(sm) - 1;
            sm &= sm - 1;
            float mine = x[0];
#pragma unroll
            for (int q = 1; q < 8; ++q)
              if (e == q) mine = x[q];
            const float cv = __shfl_sync(0xffffffffu, mine, src);
            const int ci = sg + e;
            if (better(cv, ci, fv, fi)) {  // the floor may have risen since the masks
              wt.insert(cv, ci, lane);
              // the floor only rises: the list's KM-th entry once it beats the seed
              const float nv = __shfl_sync(0xffffffffu, wt.v, KM - 1);
              const int ni = __shfl_sync(0xffffffffu, wt.i, KM - 1);
              if (better(nv, ni, fv, fi)) {
                fv = nv;
                fi = ni;
              }
            }
          }
        }
      }
    }
  }
  if constexpr (KM == 1) {
    warp_best(lv, li);
    wt.v = lv;
    wt.i = li;
  }
  __shared__ float wv[kSelWarps * KM];
  __shared__ int wi[kSelWarps * KM];
  __shared__ float smx;
  if (lane < KM) {
    wv[w * KM + lane] = wt.v;
    wi[w * KM + lane] = wt.i;
  }
  __syncthreads();
  if (w == 0) {
    int pos = 0;
    const int rounds = k < 1 ? 1 : k;
    for (int r = 0; r < rounds; ++r) {
      float bv = lane < kSelWarps && pos < KM ? wv[lane * KM + pos] : -INFINITY;
      int bi = lane < kSelWarps && pos < KM ? wi[lane * KM + pos] : INT_MAX;
      const int mine = bi;
      warp_best(bv, bi);
      if (r == 0 && lane == 0) smx = bv;
      if (mine == bi && lane < kSelWarps) ++pos;
      if (lane == 0 && r < k) {
        ids[r] = bi;
        if (vals) vals[r] = bv;
      }
    }
  }
  __syncthreads();
  return smx;
}

template <int KM>
__device__ float row_topk(const __nv_bfloat16* row, int V, int k, int* ids, float* vals) {
  return range_topk<KM>(row, 0, V >> 3, k, ids, vals);
}

// ---------------------------------------------------------------- cluster top-k
// A row split over a cluster of kSlices CTAs: each CTA ranks its slice, rank
// 0 merges the kSlices sorted lists read through distributed shared memory.
constexpr int kSlices = 8;

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t dsmem_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}

__device__ __forceinline__ float dsmem_ld_f32(uint32_t a) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
  return v;
}

__device__ __forceinline__ int dsmem_ld_s32(uint32_t a) {
  int v;
  asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  return v;
}

template <int KM>
__global__ void __launch_bounds__(kSelThreads) topk_cluster_kernel(const __nv_bfloat16* __restrict__ logits, int V,
                                                                   int k, int* __restrict__ ids,
                                                                   float* __restrict__ vals) {
  __shared__ int cid[kKMax];
  __shared__ float cval[kKMax];
  pdl_trigger();
  pdl_wait();
  const int row = blockIdx.y;
  const uint32_t rank = cluster_rank();
  const int ng = V >> 3;
  const int g0 = static_cast<int>(static_cast<long long>(ng) * rank / kSlices);
  const int g1 = static_cast<int>(static_cast<long long>(ng) * (rank + 1) / kSlices);
  range_topk<KM>(logits + static_cast<int64_t>(row) * V, g0, g1, k, cid, cval);
  __syncthreads();
  cluster_sync_all();
  if (rank == 0) {
    // gather every slice's sorted list with one parallel round of DSMEM loads
    __shared__ float gv[kSlices * kKMax];
    __shared__ int gi[kSlices * kKMax];
    const int t = threadIdx.x;
    if (t < kSlices * k) {
      const int c = t / k, j = t - c * k;
      gv[c * kKMax + j] = dsmem_ld_f32(dsmem_addr(cval + j, c));
      gi[c * kKMax + j] = dsmem_ld_s32(dsmem_addr(cid + j, c));
    }
    __syncthreads();
    if (t == 0) {
      int pos[kSlices];
#pragma unroll
      for (int c = 0; c < kSlices; ++c) pos[c] = 0;
      for (int r = 0; r < k; ++r) {
        int b = -1;
        float bv = -INFINITY;
        int bi = INT_MAX;
#pragma unroll
        for (int c = 0; c < kSlices; ++c) {
          if (pos[c] >= k) continue;
          const float v = gv[c * kKMax + pos[c]];
          const int i = gi[c * kKMax + pos[c]];
          if (b < 0 || better(v, i, bv, bi)) {
            b = c;
            bv = v;
            bi = i;
          }
        }
        ids[static_cast<int64_t>(row) * k + r] = bi;
        if (vals) vals[static_cast<int64_t>(row) * k + r] = bv;
        ++pos[b];
      }
    }
  }
  cluster_sync_all();  // every slice's shared memory stays alive until rank 0 has read it
}

// ---------------------------------------------------------------- merge of per-tile candidates
// Row `blockIdx.y`: `tiles` sorted lists of k (value, id) written by a GEMM
// epilogue, split over a cluster of kSlices CTAs. Thread j of a CTA keeps the
// best KM of its slice's candidates j, j + 512, ...; the CTA's top k comes
// from warp-shuffle rounds (block_topk); rank 0 merges the kSlices sorted
// lists read through distributed shared memory (larger value, then lower id).
template <int KM>
__global__ void __launch_bounds__(kSelThreads) topk_merge_kernel(const float* __restrict__ cand_v,
                                                                 const int* __restrict__ cand_i, int tiles, int k,
                                                                 int* __restrict__ ids, float* __restrict__ vals) {
  __shared__ int cid[kKMax];
  __shared__ float cval[kKMax];
  __shared__ float wv[kSelWarps * KM];
  __shared__ int wi[kSelWarps * KM];
  pdl_trigger();
  pdl_wait();
  const int row = blockIdx.y;
  const uint32_t rank = cluster_rank();
  const int n = tiles * k;
  const int c_begin = static_cast<int>(static_cast<long long>(n) * rank / kSlices);
  const int c_end = static_cast<int>(static_cast<long long>(n) * (rank + 1) / kSlices);
  const float* cv = cand_v + static_cast<int64_t>(row) * n;
  const int* ci = cand_i + static_cast<int64_t>(row) * n;
  float v[KM];
  int id[KM];
#pragma unroll
  for (int j = 0; j < KM; ++j) {
    v[j] = -INFINITY;
    id[j] = INT_MAX;
  }
  // four candidates in flight before any is ranked
  for (int c0 = c_begin + static_cast<int>(threadIdx.x); c0 < c_end; c0 += 4 * kSelThreads) {
    float x[4];
    int xi[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int c = c0 + u * kSelThreads;
      x[u] = c < c_end ? __ldcg(cv + c) : -INFINITY;
      xi[u] = c < c_end ? __ldcg(ci + c) : INT_MAX;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) list_insert<KM>(v, id, x[u], xi[u]);
  }
  block_topk<KM>(v, id, k, cid, cval, wv, wi);
  cluster_sync_all();
  if (rank == 0) {
    __shared__ float gv[kSlices * kKMax];
    __shared__ int gi[kSlices * kKMax];
    const int t = threadIdx.x;
    if (t < kSlices * k) {
      const int c = t / k, j = t - c * k;
      gv[c * kKMax + j] = dsmem_ld_f32(dsmem_addr(cval + j, c));
      gi[c * kKMax + j] = dsmem_ld_s32(dsmem_addr(cid + j, c));
    }
    __syncthreads();
    if (t < 32) {
      // lane c walks slice c's list; k rounds of a warp arg-max
      int pos = 0;
      for (int r = 0; r < k; ++r) {
        float bv = t < kSlices && pos < k ? gv[t * kKMax + pos] : -INFINITY;
        int bi = t < kSlices && pos < k ? gi[t * kKMax + pos] : INT_MAX;
        const int mine = bi;
        warp_best(bv, bi);
        if (mine == bi && t < kSlices) ++pos;
        if (t == 0) {
          ids[static_cast<int64_t>(row) * k + r] = bi;
          if (vals) vals[static_cast<int64_t>(row) * k + r] = bv;
        }
      }
    }
  }
  cluster_sync_all();  // every slice's shared memory stays alive until rank 0 has read it
}

template <int KM>
cudaError_t launch_topk_cluster(const __nv_bfloat16* logits, int rows, int V, int k, int* ids, float* vals,
                                cudaStream_t st) {
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kSlices;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(kSlices, rows);
  cfg.blockDim = dim3(kSelThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, topk_cluster_kernel<KM>, logits, V, k, ids, vals);
}

// 2^x by the SFU's approximate base-2 exponential (relative error a few
// units of fp32's last place; -inf gives +0).
__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Weight of id j for inverse-CDF draws; `mode` 0: exp((x - mx) / T) of one
// row; mode 1: max(p - q, 0) of two rows with their (max, sum).
struct Weights {
  const __nv_bfloat16* a;
  const __nv_bfloat16* b;
  float ma, sa, mb, sb, invT;
  int mode;
  // exp((x - m) / T) as 2^(x k - m k) with k = log2(e) / T: one fused
  // multiply-add and the SFU's base-2 exponential a value; the row sums
  // divide through reciprocals
  __device__ __forceinline__ void eval8(int g, float (&w)[8]) const {
    const float k = invT * 1.4426950408889634f;
    float x[8];
    load8(a, g, x);
    if (mode == 0) {
      const float c = -ma * k;
#pragma unroll
      for (int e = 0; e < 8; ++e) w[e] = ex2f(fmaf(x[e], k, c));
    } else {
      float y[8];
      load8(b, g, y);
      const float ca = -ma * k, cb = -mb * k;
      const float ra = 1.f / sa, rb = 1.f / sb;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        // p and q rounded on their own (__fmul_rn is never fused into the
        // subtraction): equal rows give a residual of exactly zero
        const float p = __fmul_rn(ex2f(fmaf(x[e], k, ca)), ra);
        const float q = __fmul_rn(ex2f(fmaf(y[e], k, cb)), rb);
        w[e] = fmaxf(p - q, 0.f);
      }
    }
  }
};

__device__ __forceinline__ float warp_incl_scan(float v, int lane) {
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float o = __shfl_up_sync(0xffffffffu, v, off);
    if (lane >= off) v += o;
  }
  return v;
}

// Warp w's contiguous piece of the 8-element groups [gb, ge).
__device__ __forceinline__ Slice range_slice(int gb, int ge, int w) {
  const int ng = ge - gb;
  return {gb + static_cast<int>(static_cast<long long>(ng) * w / kSelWarps),
          gb + static_cast<int>(static_cast<long long>(ng) * (w + 1) / kSelWarps)};
}

// Sum of the weights of the groups [gb, ge) in the fixed scan order (each
// warp its piece, lanes interleaved); every thread gets the total.
__device__ float weights_total(const Weights& W, int gb, int ge, float* sw) {
  __syncthreads();  // sw may still be read by a previous total / draw
  const int w = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const Slice sl = range_slice(gb, ge, w);
  float run = 0.f;
  for (int g0 = sl.g0; g0 < sl.g1; g0 += 32) {
    const int g = g0 + lane;
    float s8 = 0.f;
    if (g < sl.g1) {
      float x[8];
      W.eval8(g, x);
#pragma unroll
      for (int e = 0; e < 8; ++e) s8 += x[e];
    }
    const float inc = warp_incl_scan(s8, lane);
    run += __shfl_sync(0xffffffffu, inc, 31);
  }
  if (lane == 0) sw[w] = run;
  __syncthreads();
  float tot = 0.f;
  for (int j = 0; j < kSelWarps; ++j) tot += sw[j];
  return tot;  // sw[] stays valid for weights_draw
}
__device__ float weights_total(const Weights& W, int V, float* sw) { return weights_total(W, 0, V >> 3, sw); }

// Smallest id whose running sum exceeds thr, summed in the order of
// weights_total (which must have filled sw). Lane ranges inside a step are
// [B_{L-1}, B_L) with B_L = run + inclusive_scan_L, computed the same way for
// every lane, so they tile the step exactly. Rounding can still leave thr at
// or past the end of a slice or a lane; the draw then falls back to the last
// id with positive weight there.
__device__ int weights_draw(const Weights& W, int gb, int ge, float thr, const float* sw, int* sres) {
  const int w = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) sres[0] = -1;
  float pre = 0.f;
  int ws = -1;
  float tl = 0.f;
  for (int j = 0; j < kSelWarps; ++j) {
    const float t = thr - pre;
    if (t < sw[j] && sw[j] > 0.f) {
      ws = j;
      tl = t;
      break;
    }
    pre += sw[j];
  }
  if (ws < 0) {
    for (int j = kSelWarps - 1; j >= 0 && ws < 0; --j)
      if (sw[j] > 0.f) ws = j;
    tl = INFINITY;
  }
  __syncthreads();
  if (w == ws) {
    const Slice sl = range_slice(gb, ge, w);
    float run = 0.f;
    int last_pos = -1;
    bool done = false;
    for (int g0 = sl.g0; g0 < sl.g1 && !done; g0 += 32) {
      const int g = g0 + lane;
      float x[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = 0.f;
      float s8 = 0.f;
      if (g < sl.g1) {
        W.eval8(g, x);
#pragma unroll
        for (int e = 0; e < 8; ++e) s8 += x[e];
      }
      const float inc = warp_incl_scan(s8, lane);
      const float tot = __shfl_sync(0xffffffffu, inc, 31);
      int lp = -1;
#pragma unroll
      for (int e = 0; e < 8; ++e)
        if (x[e] > 0.f) lp = g * 8 + e;
      for (int off = 16; off >= 1; off >>= 1) lp = max(lp, __shfl_xor_sync(0xffffffffu, lp, off));
      if (lp >= 0) last_pos = lp;
      if (tl < run + tot) {
        const float B = run + inc;
        float Bp = __shfl_up_sync(0xffffffffu, B, 1);
        const bool mine = (lane == 0 || tl >= Bp) && tl < B;
        const unsigned who = __ballot_sync(0xffffffffu, mine);
        const int src = __ffs(who) - 1;  // who != 0: lane 31 has B = run + tot > tl
        if (lane == src) {
          float c = lane == 0 ? run : Bp;
          int pick = -1, lastp = -1;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            if (x[e] > 0.f) lastp = g * 8 + e;
            c += x[e];
            if (pick < 0 && tl < c && x[e] > 0.f) pick = g * 8 + e;
          }
          if (pick < 0) pick = lastp >= 0 ? lastp : last_pos;
          sres[0] = pick;
        }
        done = true;
      }
      run += tot;
    }
    __syncwarp();
    if (lane == 0 && sres[0] < 0) sres[0] = last_pos >= 0 ? last_pos : 0;
  }
  __syncthreads();
  const int r = sres[0];
  __syncthreads();
  return r;
}
__device__ int weights_draw(const Weights& W, int V, float thr, const float* sw, int* sres) {
  return weights_draw(W, 0, V >> 3, thr, sw, sres);
}

// One CTA a row: the top-k (k <= KM) of the row and, with uniforms, one
// inverse-CDF draw from softmax(row / T).
template <int KM>
__global__ void __launch_bounds__(kSelThreads) topk_kernel(const __nv_bfloat16* __restrict__ logits, int V, int k,
                                                           float invT, const float* __restrict__ uniforms,
                                                           int* __restrict__ ids, float* __restrict__ vals,
                                                           int* __restrict__ sampled) {
  pdl_trigger();
  pdl_wait();
  __shared__ float sw[kSelWarps];
  __shared__ int sres[1];
  __shared__ int sid[kKMax];
  __shared__ float sval[kKMax];
  const int r = blockIdx.x;
  const __nv_bfloat16* row = logits + static_cast<int64_t>(r) * V;
  const float mx = row_topk<KM>(row, V, k, sid, sval);
  __syncthreads();
  if (threadIdx.x < k) {
    ids[static_cast<int64_t>(r) * k + threadIdx.x] = sid[threadIdx.x];
    if (vals) vals[static_cast<int64_t>(r) * k + threadIdx.x] = sval[threadIdx.x];
  }
  if (uniforms != nullptr) {
    Weights W{row, nullptr, mx, 1.f, 0.f, 1.f, invT, 0};
    const float tot = weights_total(W, V, sw);
    const int j = weights_draw(W, V, uniforms[r] * tot, sw, sres);
    if (threadIdx.x == 0) sampled[r] = j;
  }
}

// greedy, step 1 (t_i = argmax of every target row -> out[s][i]) is the
// cluster top-k with k = 1.

// greedy, step 2: longest prefix of drafts equal to the target argmax, then
// the bonus token; rewrites out[s][*] in place.
__global__ void greedy_prefix_kernel(int S, int V, const int* __restrict__ draft, int dld,
                                     int* __restrict__ accept, int* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= S) return;
  // every load issued before the first comparison (no chain of dependent loads)
  int t[16], d[15];
#pragma unroll
  for (int i = 0; i < 16; ++i) t[i] = out[s * 16 + i];
#pragma unroll
  for (int i = 0; i < 15; ++i) d[i] = draft[(s * 15 + i) * dld];
  int a = 15;
#pragma unroll
  for (int i = 14; i >= 0; --i)
    if (d[i] != t[i]) a = i;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    int v = -1;
    if (i < a) v = d[i];
    if (i == a) v = t[i];
    out[s * 16 + i] = v;
  }
  accept[s] = a;
}

// sampling, step 1: (max, sum of exp((x - max) / T)) of every target row
// (r < 16) and draft row (r >= 16) of a stream in one pass: every thread
// keeps a running (max, sum) over its 8-element groups (rescaled when the
// max moves), merged over the warp by a xor tree and over the warps in
// order.
__device__ __forceinline__ void ms_merge2(float& m, float& sum, float m2, float s2, float k) {
  const float mm = fmaxf(m, m2);
  const float a = m == -INFINITY ? 0.f : sum * ex2f((m - mm) * k);
  const float b = m2 == -INFINITY ? 0.f : s2 * ex2f((m2 - mm) * k);
  m = mm;
  sum = a + b;
}

__global__ void __launch_bounds__(kSelThreads) softmax_stats_kernel(const __nv_bfloat16* __restrict__ tl,
                                                                    const __nv_bfloat16* __restrict__ dl, int V,
                                                                    float invT, float* __restrict__ stats) {
  pdl_trigger();
  pdl_wait();
  __shared__ float wm[kSelWarps], wsum[kSelWarps];
  const int r = blockIdx.x;
  const int s = blockIdx.y;
  const __nv_bfloat16* row =
      r < 16 ? tl + (static_cast<int64_t>(s) * 16 + r) * V : dl + (static_cast<int64_t>(s) * 15 + (r - 16)) * V;
  const float k = invT * 1.4426950408889634f;
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Slice sl = warp_slice(V, w);
  float m = -INFINITY, sum = 0.f;
  for (int g0 = sl.g0 + lane; g0 < sl.g1; g0 += 4 * 32) {
    uint4 raw[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int g = g0 + u * 32;
      raw[u] = g < sl.g1 ? *reinterpret_cast<const uint4*>(row + static_cast<int64_t>(g) * 8)
                         : make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);  // bf16 -inf
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float gm = max8(raw[u]);
      if (gm == -INFINITY) continue;
      const float nm = fmaxf(m, gm);
      if (nm > m) {
        sum = m == -INFINITY ? 0.f : sum * ex2f((m - nm) * k);
        m = nm;
      }
      float x[8];
      unpack8(raw[u], x);
      const float c = -m * k;
#pragma unroll
      for (int e = 0; e < 8; ++e) sum += ex2f(fmaf(x[e], k, c));
    }
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
    const float s2 = __shfl_xor_sync(0xffffffffu, sum, off);
    ms_merge2(m, sum, m2, s2, k);
  }
  if (lane == 0) {
    wm[w] = m;
    wsum[w] = sum;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float M = wm[0], Sm = wsum[0];
    for (int j = 1; j < kSelWarps; ++j) ms_merge2(M, Sm, wm[j], wsum[j], k);
    stats[(s * 31 + r) * 2] = M;
    stats[(s * 31 + r) * 2 + 1] = Sm;
  }
}

// sampling, step 2: the accept chain (every CTA of the stream's cluster
// takes it), then the residual or bonus draw with the row split over the
// kSlices CTAs: each sums the weights of its slice, the slice sums meet
// through distributed shared memory (added in rank order), and the CTA
// whose slice holds the threshold draws within it.
__global__ void __launch_bounds__(kSelThreads) sample_verify_kernel(int V, const int* __restrict__ draft, int dld,
                                                                    const __nv_bfloat16* __restrict__ tl,
                                                                    const __nv_bfloat16* __restrict__ dl,
                                                                    const float* __restrict__ u, float invT,
                                                                    const float* __restrict__ stats,
                                                                    int* __restrict__ accept, int* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  __shared__ float sw[kSelWarps];
  __shared__ int sres[1];
  __shared__ float slice_tot[2];  // read by the other CTAs of the cluster
  __shared__ int rejected[16];
  const uint32_t rank = cluster_rank();
  const int s = blockIdx.y;
  const float* st = stats + s * 31 * 2;
  // the 15 acceptance tests at once, thread i taking position i (their
  // loads in parallel, not a chain); a = the first rejected position
  if (threadIdx.x < 15) {
    const int i = threadIdx.x;
    const int x = draft[(s * 15 + i) * dld];
    bool acc = false;
    if (x >= 0 && x < V) {
      const float p = expf((__bfloat162float(tl[(static_cast<int64_t>(s) * 16 + i) * V + x]) - st[i * 2]) * invT) /
                      st[i * 2 + 1];
      const float q =
          expf((__bfloat162float(dl[(static_cast<int64_t>(s) * 15 + i) * V + x]) - st[(16 + i) * 2]) * invT) /
          st[(16 + i) * 2 + 1];
      acc = u[(s * 16 + i) * 2] * q < p;
    }
    rejected[i] = acc ? 0 : 1;
  }
  __syncthreads();
  int a = 15;
  for (int i = 14; i >= 0; --i)
    if (rejected[i]) a = i;
  const int ng = V >> 3;
  const int gb = static_cast<int>(static_cast<long long>(ng) * rank / kSlices);
  const int ge = static_cast<int>(static_cast<long long>(ng) * (rank + 1) / kSlices);
  const __nv_bfloat16* trow = tl + (static_cast<int64_t>(s) * 16 + a) * V;
  const float ud = u[(s * 16 + a) * 2 + 1];
  Weights W{trow, nullptr, st[a * 2], 1.f, 0.f, 1.f, invT, 0};
  if (a < 15)
    W = Weights{trow, dl + (static_cast<int64_t>(s) * 15 + a) * V, st[a * 2], st[a * 2 + 1], st[(16 + a) * 2],
                st[(16 + a) * 2 + 1], invT, 1};
  // the slice sums of the cluster, in rank order
  float tots[kSlices];
  float total = 0.f;
  for (int pass = 0; pass < 2; ++pass) {
    const float t = weights_total(W, gb, ge, sw);
    if (threadIdx.x == 0) slice_tot[pass] = t;
    cluster_sync_all();
    total = 0.f;
#pragma unroll
    for (int r2 = 0; r2 < kSlices; ++r2) {
      tots[r2] = dsmem_ld_f32(dsmem_addr(&slice_tot[pass], r2));
      total += tots[r2];
    }
    // an all-zero residual: draw from the target's distribution instead
    if (total > 0.f || W.mode == 0) break;
    W = Weights{trow, nullptr, st[a * 2], 1.f, 0.f, 1.f, invT, 0};
  }
  const float thr = ud * total;
  int js = -1;
  float pre = 0.f, tin = 0.f;
  for (int r2 = 0; r2 < kSlices; ++r2) {
    if (thr - pre < tots[r2] && tots[r2] > 0.f) {
      js = r2;
      tin = thr - pre;
      break;
    }
    pre += tots[r2];
  }
  if (js < 0) {  // rounding left the threshold past the end: the last slice with weight
    for (int r2 = kSlices - 1; r2 >= 0 && js < 0; --r2)
      if (tots[r2] > 0.f) js = r2;
    if (js < 0) js = 0;  // no weight anywhere: rank 0's draw returns id 0
    tin = INFINITY;
  }
  if (static_cast<int>(rank) == js) {
    const int tok = weights_draw(W, gb, ge, tin, sw, sres);
    if (threadIdx.x == 0) out[s * 16 + a] = tok;
  }
  if (rank == 0) {
    if (threadIdx.x < 16 && threadIdx.x != a) {
      const int i = threadIdx.x;
      out[s * 16 + i] = i < a ? draft[(s * 15 + i) * dld] : -1;
    }
    if (threadIdx.x == 0) accept[s] = a;
  }
  cluster_sync_all();  // the slice sums stay alive until every rank has read them
}

}  // namespace

// ---------------------------------------------------------------- confidence and min-p stop
// conf[r] = the largest entry of softmax(row r / T) = 1 / sum_j exp((x_j - max) / T):
// one CTA a row, one pass; every thread keeps a running (max, sum) over its
// 8-element groups, the pairs merge by a xor tree in each warp and then over
// the warps in order (the element equal to the final max contributes 1).
__device__ __forceinline__ void ms_merge(float& m, float& s, float m2, float s2, float invT) {
  const float mm = fmaxf(m, m2);
  const float a = m == -INFINITY ? 0.f : s * expf((m - mm) * invT);
  const float b = m2 == -INFINITY ? 0.f : s2 * expf((m2 - mm) * invT);
  m = mm;
  s = a + b;
}

__global__ void __launch_bounds__(kSelThreads) conf_kernel(const __nv_bfloat16* __restrict__ logits, int V,
                                                           float invT, float* __restrict__ conf) {
  __shared__ float wm[kSelWarps], ws[kSelWarps];
  pdl_trigger();
  pdl_wait();
  const int r = blockIdx.x;
  const __nv_bfloat16* row = logits + static_cast<int64_t>(r) * V;
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Slice sl = warp_slice(V, w);
  float m = -INFINITY, sm = 0.f;
  for (int g0 = sl.g0 + lane; g0 < sl.g1; g0 += 4 * 32) {
    float x[4][8];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int g = g0 + u * 32;
      if (g < sl.g1) {
        load8(row, g, x[u]);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) x[u][e] = -INFINITY;
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      float gm = x[u][0];
#pragma unroll
      for (int e = 1; e < 8; ++e) gm = fmaxf(gm, x[u][e]);
      if (gm == -INFINITY) continue;
      float gs = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) gs += expf((x[u][e] - gm) * invT);
      ms_merge(m, sm, gm, gs, invT);
    }
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
    const float s2 = __shfl_xor_sync(0xffffffffu, sm, off);
    ms_merge(m, sm, m2, s2, invT);
  }
  if (lane == 0) {
    wm[w] = m;
    ws[w] = sm;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float M = wm[0], S = ws[0];
    for (int j = 1; j < kSelWarps; ++j) ms_merge(M, S, wm[j], ws[j], invT);
    conf[r] = 1.f / S;
  }
}

// len[s] = the number of leading rows of stream s (15 a stream) whose
// confidence is at least min_p.
__global__ void stop_len_kernel(const float* __restrict__ conf, int S, float min_p, int* __restrict__ len) {
  pdl_trigger();
  pdl_wait();
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= S) return;
  int n = 0;
  while (n < 15 && conf[s * 15 + n] >= min_p) ++n;
  len[s] = n;
}

int launch_draft_stop(const __nv_bfloat16* logits, int streams, int V, float T, float min_p, float* conf, int* len,
                      cudaStream_t st) {
  if (streams <= 0) return DFLASH_OK;
  {
    TraceScope ts(st, "draft_stop.conf", static_cast<double>(streams) * 15 * V * 2, 0.0);
    const cudaError_t e = launch_pdl(conf_kernel, dim3(streams * 15), dim3(kSelThreads), 0, st, logits, V, 1.0f / T, conf);
    count_launch();
    if (e != cudaSuccess) return DFLASH_E_CUDA;
  }
  {
    TraceScope ts(st, "draft_stop.len", static_cast<double>(streams) * 15 * 4, 0.0);
    const cudaError_t e =
        launch_pdl(stop_len_kernel, dim3((streams + 127) / 128), dim3(128), 0, st, conf, streams, min_p, len);
    count_launch();
    if (e != cudaSuccess) return DFLASH_E_CUDA;
  }
  return DFLASH_OK;
}

int launch_topk_merge(const float* cand_v, const int* cand_i, int rows, int tiles, int k, int* ids, float* vals,
                      cudaStream_t st) {
  if (rows <= 0) return DFLASH_OK;
  if (k < 1 || k > 8) return DFLASH_E_INVALID_ARG;
  TraceScope ts(st, "topk_merge", static_cast<double>(rows) * tiles * k * 8, 0.0);
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kSlices;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(kSlices, rows);
  cfg.blockDim = dim3(kSelThreads);
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, topk_merge_kernel<8>, cand_v, cand_i, tiles, k, ids, vals);
  count_launch();
  return cuda_status(e);
}

// Plain top-k scans: up to kClusterRows rows a row is split over a cluster of
// kSlices CTAs (few rows: fill the GPU); more rows already fill it, and one
// CTA a row avoids the cluster's fixed ranking and merge cost per slice. The
// ranking is exact with ties to the lower id, so both give the same result.
constexpr int kClusterRows = 64;

template <int KM>
cudaError_t launch_topk_scan(const __nv_bfloat16* logits, int rows, int V, int k, int* ids, float* vals,
                             cudaStream_t st) {
  if (rows <= kClusterRows) return launch_topk_cluster<KM>(logits, rows, V, k, ids, vals, st);
  return launch_pdl(topk_kernel<KM>, dim3(rows), dim3(kSelThreads), 0, st, logits, V, k, 1.0f, nullptr, ids, vals,
                    nullptr);
}

int launch_topk(const __nv_bfloat16* logits, int rows, int V, int k, float T, const float* uniforms, int* ids,
                float* vals, int* sampled, cudaStream_t st) {
  if (rows <= 0) return DFLASH_OK;
  TraceScope ts(st, "topk", static_cast<double>(rows) * V * 2, 0.0);
  cudaError_t e;
  if (uniforms == nullptr && k >= 1) {
    // k = 1 takes the lanes' own running arg-max (one compare-select a
    // value, one warp reduction at the end) instead of the warp lists
    e = k == 1   ? launch_topk_scan<1>(logits, rows, V, k, ids, vals, st)
        : k <= 8 ? launch_topk_scan<8>(logits, rows, V, k, ids, vals, st)
                 : launch_topk_scan<kKMax>(logits, rows, V, k, ids, vals, st);
  } else if (k <= 8) {
    e = launch_pdl(topk_kernel<8>, dim3(rows), dim3(kSelThreads), 0, st, logits, V, k, 1.0f / T, uniforms, ids, vals,
                   sampled);
  } else {
    e = launch_pdl(topk_kernel<kKMax>, dim3(rows), dim3(kSelThreads), 0, st, logits, V, k, 1.0f / T, uniforms, ids,
                   vals, sampled);
  }
  count_launch();
  return cuda_status(e);
}

int launch_verify_greedy(int S, int V, const int* draft, int dld, const __nv_bfloat16* tl, int* accept, int* out,
                         cudaStream_t st) {
  {
    TraceScope ts(st, "verify.argmax", static_cast<double>(S) * 16 * V * 2, 0.0);
    const cudaError_t e = launch_topk_scan<1>(tl, S * 16, V, 1, out, nullptr, st);
    count_launch();
    if (e != cudaSuccess) return DFLASH_E_CUDA;
  }
  {
    TraceScope ts(st, "verify.prefix", S * 31.0 * 4, 0.0);
    const cudaError_t e =
        launch_pdl(greedy_prefix_kernel, dim3((S + 127) / 128), dim3(128), 0, st, S, V, draft, dld, accept, out);
    count_launch();
    if (e != cudaSuccess) return DFLASH_E_CUDA;
  }
  return cuda_status(cudaGetLastError());
}

int launch_verify_sample(int S, int V, const int* draft, int dld, const __nv_bfloat16* tl, const __nv_bfloat16* dl,
                         const float* u, float T, int* accept, int* out, float* stats, cudaStream_t st) {
  dim3 g(31, S);
  {
    TraceScope ts(st, "verify.softmax_stats", static_cast<double>(S) * 31 * V * 2, 0.0);
    const cudaError_t e = launch_pdl(softmax_stats_kernel, g, dim3(kSelThreads), 0, st, tl, dl, V, 1.0f / T, stats);
    count_launch();
    if (e != cudaSuccess) return DFLASH_E_CUDA;
  }
  {
    TraceScope ts(st, "verify.sample", static_cast<double>(S) * 2 * V * 2, 0.0);
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kSlices;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(kSlices, S);
    cfg.blockDim = dim3(kSelThreads);
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, sample_verify_kernel, V, draft, dld, tl, dl, u, 1.0f / T,
                                             static_cast<const float*>(stats), accept, out);
    count_launch();
    if (e != cudaSuccess) return DFLASH_E_CUDA;
  }
  return cuda_status(cudaGetLastError());
}

}  // namespace dfl
