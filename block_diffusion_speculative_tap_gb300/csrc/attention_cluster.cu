// Block attention for head dimension 128 as one thread-block cluster per
// (stream, kv head).
//
// The visible context keys of a (stream, kv head) are split evenly over the
// CS CTAs of a cluster (8; 4 or 2 when many streams already fill the GPU);
// the last CTA also takes the block's own 16 rows. When the query heads of a kv head are an even number, two clusters
// share the kv head, each taking half of its query heads (K/V tiles are read
// by both, the second read mostly from L2), so twice as many SMs stream.
// Inside a CTA one producer thread streams 64-key tiles of K and V from the
// head-major cache with TMA (3-D tensor maps, 128-byte swizzle) through a
// ring of kStages shared-memory stages; 2G consumer warps (G = query heads
// of the CTA, two key-tile parities each) compute scores and P*V on the
// tensor cores (mma.sync m16n8k16, P in bf16) with an online softmax. The two parities of a head merge in shared memory, then the CTAs
// of the cluster reduce-scatter their partial (max, sum, output) through
// distributed shared memory, in rank order, and write the bf16 attention
// output: no partials in global memory and no second kernel. Up to four
// streams a launch the split is always 8 ways and depends only on the
// stream's visible length, so a stream's result does not depend on the batch.
#include <mutex>
#include <utility>
#include <vector>

#include "internal.h"
#include "ptx.cuh"

namespace dfl {

namespace {

constexpr int kD = 128;
constexpr int kKeys = 64;             // keys per context tile
constexpr int kBlockKeys = 16;        // the block's own keys
constexpr int kStages = 3;
constexpr int kClusterCtas = 8;  // CTAs a cluster up to four streams a launch
constexpr int kSubBytes = kKeys * 128;   // 64 rows x 64 dims (128 B) per swizzled sub-tile
constexpr int kTileBytes = 4 * kSubBytes;  // K lo, K hi, V lo, V hi = 32 KiB
constexpr int kBlockSubBytes = kBlockKeys * 128;
constexpr int kPartLd = kD + 8;       // fp32 partial row stride (conflict-free float2 stores)

// Under 113 KiB, so two CTAs fit an SM and a cluster of 8 spans four SMs.
struct ClusterAttnSmem {
  static constexpr int kStageOff = 0;
  static constexpr int kBlockOff = kStages * kTileBytes;       // block tile: 16 keys
  static constexpr int kBarOff = kBlockOff + 4 * kBlockSubBytes;
  static constexpr int kBytes = kBarOff + 8 * (2 * kStages + 1) + 64;
};

__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t saddr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(saddr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t saddr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(saddr));
}

// P (probabilities in [0, 1]) enters P*V as bf16; the row sum l uses the
// unrounded fp32 values.
__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Byte offset of (row, 16-byte chunk) in a 128-byte-swizzled sub-tile.
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ void tma3d(uint32_t dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

__device__ __forceinline__ void tma2d(uint32_t dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}

__device__ __forceinline__ uint32_t crank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void csync() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
__device__ __forceinline__ uint32_t cmap(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ float cld(uint32_t a) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ float4 cld4(uint32_t a) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(a)
               : "memory");
  return v;
}

struct AttnState {
  float o[kD / 8][4];
  float m[2];
  float l[2];
};

// One tile of NK keys at shared address `t` (K lo/hi, V lo/hi sub-tiles of
// NK rows each) for keys [0, nvalid); scores use `sc` = log2(e) / sqrt(d).
template <int NK>
__device__ __forceinline__ void attend_tile(AttnState& S, const uint32_t (&qa)[kD / 16][4], uint32_t t, int nvalid,
                                            float sc, int lane) {
  constexpr uint32_t kSub = NK * 128;
  constexpr int kN = NK / 8;  // 8-key score tiles
  float sacc[kN][4];
#pragma unroll
  for (int n = 0; n < kN; ++n) sacc[n][0] = sacc[n][1] = sacc[n][2] = sacc[n][3] = 0.f;
  // Each score tile accumulates its 8 k16 steps in order; the MMAs issue
  // over groups of up to four score tiles, so consecutive MMAs are
  // independent (a tile's own chain would wait out each MMA's latency).
  constexpr int kGrp = kN < 4 ? kN : 4;
#pragma unroll
  for (int n0 = 0; n0 < kN; n0 += kGrp) {
#pragma unroll
    for (int kp = 0; kp < kD / 32; ++kp) {
      // four 8x8 matrices a tile: dims [32kp, 32kp + 32) of keys n*8 .. n*8+7
      uint32_t kb[kGrp][4];
#pragma unroll
      for (int g = 0; g < kGrp; ++g)
        ldsm_x4(kb[g], t + static_cast<uint32_t>((kp >> 1) * kSub) +
                           swz((n0 + g) * 8 + (lane & 7), 4 * (kp & 1) + (lane >> 3)));
#pragma unroll
      for (int g = 0; g < kGrp; ++g) mma16816(sacc[n0 + g], qa[2 * kp], kb[g][0], kb[g][1]);
#pragma unroll
      for (int g = 0; g < kGrp; ++g) mma16816(sacc[n0 + g], qa[2 * kp + 1], kb[g][2], kb[g][3]);
    }
  }
  float tmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
  for (int n = 0; n < kN; ++n) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int key = n * 8 + (lane & 3) * 2 + (e & 1);
      const float v = key < nvalid ? sacc[n][e] * sc : -INFINITY;
      sacc[n][e] = v;
      tmax[e >> 1] = fmaxf(tmax[e >> 1], v);
    }
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    tmax[r] = fmaxf(tmax[r], __shfl_xor_sync(0xffffffffu, tmax[r], 1));
    tmax[r] = fmaxf(tmax[r], __shfl_xor_sync(0xffffffffu, tmax[r], 2));
  }
  float mnew[2], alpha[2], psum[2] = {0.f, 0.f};
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    mnew[r] = fmaxf(S.m[r], tmax[r]);
    alpha[r] = mnew[r] == -INFINITY ? 1.f : exp2f(S.m[r] - mnew[r]);
    S.m[r] = mnew[r];
  }
#pragma unroll
  for (int n = 0; n < kN; ++n) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float p = mnew[e >> 1] == -INFINITY ? 0.f : exp2f(sacc[n][e] - mnew[e >> 1]);
      sacc[n][e] = p;
      psum[e >> 1] += p;
    }
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    psum[r] += __shfl_xor_sync(0xffffffffu, psum[r], 1);
    psum[r] += __shfl_xor_sync(0xffffffffu, psum[r], 2);
    S.l[r] = S.l[r] * alpha[r] + psum[r];
  }
#pragma unroll
  for (int n = 0; n < kD / 8; ++n) {
    S.o[n][0] *= alpha[0];
    S.o[n][1] *= alpha[0];
    S.o[n][2] *= alpha[1];
    S.o[n][3] *= alpha[1];
  }
#pragma unroll
  for (int kk = 0; kk < NK / 16; ++kk) {
    uint32_t ph[4];
    ph[0] = pack_bf16(sacc[2 * kk][0], sacc[2 * kk][1]);
    ph[1] = pack_bf16(sacc[2 * kk][2], sacc[2 * kk][3]);
    ph[2] = pack_bf16(sacc[2 * kk + 1][0], sacc[2 * kk + 1][1]);
    ph[3] = pack_bf16(sacc[2 * kk + 1][2], sacc[2 * kk + 1][3]);
    const int mi = lane >> 3;
    const int key = kk * 16 + (mi & 1) * 8 + (lane & 7);
#pragma unroll
    for (int n2 = 0; n2 < kD / 16; ++n2) {
      const int dim = n2 * 16 + (mi >> 1) * 8;
      const uint32_t sub = t + static_cast<uint32_t>((2 + (dim >> 6)) * kSub);
      uint32_t vb[4];
      ldsm_x4_trans(vb, sub + swz(key, (dim & 63) >> 3));
      mma16816(S.o[2 * n2], ph, vb[0], vb[1]);
      mma16816(S.o[2 * n2 + 1], ph, vb[2], vb[3]);
    }
  }
}

struct ClusterAttnArgs {
  CUtensorMap kmap;  // cache K: 3-D [S*nkv][cap][128], box {64, 64, 1}
  CUtensorMap vmap;
  CUtensorMap kbmap;  // block K: 2-D [T][nkv*128], box {64, 16}
  CUtensorMap vbmap;
  AttnArgs a;
};

// G: query heads handled by this CTA (of the kv head's group); HS: CTAs
// (clusters) sharing a kv head; CS: CTAs a cluster, splitting the keys.
template <int G, int HS, int CS>
__global__ void __launch_bounds__(32 * (2 * G + 1), G <= 2 ? 2 : 1) attn_cluster_kernel(const __grid_constant__ ClusterAttnArgs P) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const AttnArgs& a = P.a;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + ClusterAttnSmem::kBarOff);
  uint64_t* empty = full + kStages;
  uint64_t* blkbar = empty + kStages;
  const uint32_t sbase = smem_u32(smem);

  const int ncons = 2 * G;  // consumer warps
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = crank();
  const int kvh = blockIdx.y / HS;
  const int hs = blockIdx.y - kvh * HS;
  const int head0 = kvh * (G * HS) + hs * G;  // first query head of this CTA
  const int si = blockIdx.z;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], G);
    }
    mbar_init(blkbar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  pdl_trigger();
  // The context K/V tiles and the stream lengths come from earlier fills,
  // complete before a draft call's first kernel starts (that kernel is
  // launched without programmatic dependence, or after a memset): the
  // producer loads the first stages before the PDL wait. Q and the block's
  // own K/V come from the Q/K/V GEMM, after it.
  const bool producer = warp == 2 * G && lane == 0;
  if (!producer) pdl_wait();

  const int s = a.s_begin + si;
  const int C = a.lens[s];
  const int nvis = a.window > 0 ? min(C, a.window) : C;
  const int k0 = static_cast<int>(static_cast<long long>(nvis) * rank / CS);
  const int k1 = static_cast<int>(static_cast<long long>(nvis) * (rank + 1) / CS);
  const int nt = (k1 - k0 + kKeys - 1) / kKeys;
  const bool has_block = rank == CS - 1;
  const int slab = s * a.nkv + kvh;
  int* err = a.err;

  if (warp == ncons) {
    if (lane == 0) {
      const int npre = nt < kStages ? nt : kStages;
      for (int t = 0; t < npre; ++t) {  // fresh stages: nothing to wait for
        mbar_arrive_expect_tx(&full[t], kTileBytes);
        const uint32_t d = sbase + ClusterAttnSmem::kStageOff + t * kTileBytes;
        const int row = k0 + t * kKeys;
        tma3d(d, &P.kmap, &full[t], 0, row, slab);
        tma3d(d + kSubBytes, &P.kmap, &full[t], 64, row, slab);
        tma3d(d + 2 * kSubBytes, &P.vmap, &full[t], 0, row, slab);
        tma3d(d + 3 * kSubBytes, &P.vmap, &full[t], 64, row, slab);
      }
      pdl_wait();
      if (has_block) {
        mbar_arrive_expect_tx(blkbar, 4 * kBlockSubBytes);
        const uint32_t b = sbase + ClusterAttnSmem::kBlockOff;
        tma2d(b, &P.kbmap, blkbar, kvh * kD, 16 * si);
        tma2d(b + kBlockSubBytes, &P.kbmap, blkbar, kvh * kD + 64, 16 * si);
        tma2d(b + 2 * kBlockSubBytes, &P.vbmap, blkbar, kvh * kD, 16 * si);
        tma2d(b + 3 * kBlockSubBytes, &P.vbmap, blkbar, kvh * kD + 64, 16 * si);
      }
      for (int t = npre; t < nt; ++t) {
        const int st = t % kStages;
        if (!mbar_wait(&empty[st], ((t / kStages) & 1) ^ 1u, err, DFLASH_STATUS_TIMEOUT, nullptr)) break;
        mbar_arrive_expect_tx(&full[st], kTileBytes);
        const uint32_t d = sbase + ClusterAttnSmem::kStageOff + st * kTileBytes;
        const int row = k0 + t * kKeys;
        tma3d(d, &P.kmap, &full[st], 0, row, slab);
        tma3d(d + kSubBytes, &P.kmap, &full[st], 64, row, slab);
        tma3d(d + 2 * kSubBytes, &P.vmap, &full[st], 0, row, slab);
        tma3d(d + 3 * kSubBytes, &P.vmap, &full[st], 64, row, slab);
      }
      // no copy may still be landing when the stage memory is reused below
      for (int st = 0; st < kStages && st < nt; ++st) {
        const int last = st + ((nt - 1 - st) / kStages) * kStages;
        mbar_wait(&full[st], (last / kStages) & 1, err, DFLASH_STATUS_TIMEOUT, nullptr);
      }
      if (has_block) mbar_wait(blkbar, 0, err, DFLASH_STATUS_TIMEOUT, nullptr);
    }
  }

  AttnState S;
  const int hq = warp >> 1;
  const int par = warp & 1;
  const bool consumer = warp < ncons;
  if (consumer) {
#pragma unroll
    for (int n = 0; n < kD / 8; ++n) S.o[n][0] = S.o[n][1] = S.o[n][2] = S.o[n][3] = 0.f;
    S.m[0] = S.m[1] = -INFINITY;
    S.l[0] = S.l[1] = 0.f;
    const int h = head0 + hq;
    uint32_t qa[kD / 16][4];
    {
      const __nv_bfloat16* Q = a.Q + static_cast<int64_t>(si) * 16 * (a.nq * kD) + static_cast<int64_t>(h) * kD;
      const int qr = lane >> 2, qc = (lane & 3) * 2, ld = a.nq * kD;
#pragma unroll
      for (int kk = 0; kk < kD / 16; ++kk) {
        qa[kk][0] = *reinterpret_cast<const uint32_t*>(Q + qr * ld + kk * 16 + qc);
        qa[kk][1] = *reinterpret_cast<const uint32_t*>(Q + (qr + 8) * ld + kk * 16 + qc);
        qa[kk][2] = *reinterpret_cast<const uint32_t*>(Q + qr * ld + kk * 16 + qc + 8);
        qa[kk][3] = *reinterpret_cast<const uint32_t*>(Q + (qr + 8) * ld + kk * 16 + qc + 8);
      }
    }
    const float sc = rsqrtf(static_cast<float>(kD)) * 1.4426950408889634f;
    for (int t = par; t < nt; t += 2) {
      const int st = t % kStages;
      if (!mbar_wait(&full[st], (t / kStages) & 1, err, DFLASH_STATUS_TIMEOUT, nullptr)) break;
      attend_tile<kKeys>(S, qa, sbase + ClusterAttnSmem::kStageOff + st * kTileBytes,
                         min(kKeys, k1 - k0 - t * kKeys), sc, lane);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }
    if (has_block && par == 1) {
      if (mbar_wait(blkbar, 0, err, DFLASH_STATUS_TIMEOUT, nullptr))
        attend_tile<kBlockKeys>(S, qa, sbase + ClusterAttnSmem::kBlockOff, kBlockKeys, sc, lane);
    }
  }
  __syncthreads();  // every tile consumed: the stage memory is free

  // merge the two parities of each head; the CTA partial goes to
  // part[hq][16][kPartLd] (fp32) and ml[hq][16][2], at the start of stage
  // memory; the odd-parity states pass through xch[hq][68][32] (lane-minor)
  float* part = reinterpret_cast<float*>(smem + ClusterAttnSmem::kStageOff);
  float* ml = part + G * 16 * kPartLd;
  float* xch = ml + G * 16 * 2;
  static_assert(sizeof(float) * G * (16 * (kPartLd + 2) + 68 * 32) <= kStages * kTileBytes,
                "merge scratch exceeds the stage memory");
  if (consumer && par == 1) {
    float* x = xch + hq * 68 * 32 + lane;
#pragma unroll
    for (int n = 0; n < kD / 8; ++n) {
      x[(4 * n) * 32] = S.o[n][0];
      x[(4 * n + 1) * 32] = S.o[n][1];
      x[(4 * n + 2) * 32] = S.o[n][2];
      x[(4 * n + 3) * 32] = S.o[n][3];
    }
    x[64 * 32] = S.m[0];
    x[65 * 32] = S.m[1];
    x[66 * 32] = S.l[0];
    x[67 * 32] = S.l[1];
  }
  __syncthreads();
  if (consumer && par == 0) {
    const float* x = xch + hq * 68 * 32 + lane;
    float w0[2], w1[2], M[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const float mx = x[(64 + r) * 32];
      M[r] = fmaxf(S.m[r], mx);
      w0[r] = M[r] == -INFINITY ? 0.f : exp2f(S.m[r] - M[r]);
      w1[r] = M[r] == -INFINITY ? 0.f : exp2f(mx - M[r]);
    }
    const int r0 = lane >> 2;
#pragma unroll
    for (int n = 0; n < kD / 8; ++n) {
      const int col = n * 8 + (lane & 3) * 2;
      float2* p0 = reinterpret_cast<float2*>(part + (hq * 16 + r0) * kPartLd + col);
      float2* p1 = reinterpret_cast<float2*>(part + (hq * 16 + r0 + 8) * kPartLd + col);
      *p0 = make_float2(S.o[n][0] * w0[0] + x[(4 * n) * 32] * w1[0], S.o[n][1] * w0[0] + x[(4 * n + 1) * 32] * w1[0]);
      *p1 = make_float2(S.o[n][2] * w0[1] + x[(4 * n + 2) * 32] * w1[1],
                        S.o[n][3] * w0[1] + x[(4 * n + 3) * 32] * w1[1]);
    }
    if ((lane & 3) == 0) {
      ml[(hq * 16 + r0) * 2] = M[0];
      ml[(hq * 16 + r0) * 2 + 1] = S.l[0] * w0[0] + x[66 * 32] * w1[0];
      ml[(hq * 16 + r0 + 8) * 2] = M[1];
      ml[(hq * 16 + r0 + 8) * 2 + 1] = S.l[1] * w0[1] + x[67 * 32] * w1[1];
    }
  }
  csync();  // every CTA's partial is ready

  // reduce-scatter: this rank owns (head, row) vectors [v0, v1) of the G*16
  {
    const int nvec = G * 16;
    const int v0 = static_cast<int>(rank) * nvec / CS;
    const int v1 = (static_cast<int>(rank) + 1) * nvec / CS;
    const uint32_t pbase = smem_u32(part), mlbase = smem_u32(ml);
    for (int idx = threadIdx.x; idx < (v1 - v0) * 32; idx += blockDim.x) {
      const int vec = v0 + idx / 32;
      const int d4 = (idx & 31) * 4;
      // every rank's (max, sum, partial) loaded before any is used
      float mr[CS], lr[CS];
      float4 pr[CS];
#pragma unroll
      for (int r2 = 0; r2 < CS; ++r2) {
        mr[r2] = cld(cmap(mlbase, r2) + vec * 8);
        lr[r2] = cld(cmap(mlbase, r2) + vec * 8 + 4);
        pr[r2] = cld4(cmap(pbase, r2) + (vec * kPartLd + d4) * 4);
      }
      float M = -INFINITY;
#pragma unroll
      for (int r2 = 0; r2 < CS; ++r2) M = fmaxf(M, mr[r2]);
      float den = 0.f;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int r2 = 0; r2 < CS; ++r2) {
        const float w = M == -INFINITY ? 0.f : exp2f(mr[r2] - M);
        den += w * lr[r2];
        acc.x += w * pr[r2].x;
        acc.y += w * pr[r2].y;
        acc.z += w * pr[r2].z;
        acc.w += w * pr[r2].w;
      }
      const int hq2 = vec >> 4, row = vec & 15;
      __nv_bfloat16* out =
          a.out + (static_cast<int64_t>(si) * 16 + row) * (a.nq * kD) + (head0 + hq2) * kD + d4;
      const float inv = 1.f / den;
      *reinterpret_cast<__nv_bfloat162*>(out) = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
      *reinterpret_cast<__nv_bfloat162*>(out + 2) = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
    }
  }
  csync();  // partials stay alive until every rank has read them
}

int encode_map(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
               const cuuint32_t* box) {
  using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  static EncodeFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return DFLASH_E_UNSUPPORTED;
    fn = reinterpret_cast<EncodeFn>(p);
  }
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DFLASH_OK : DFLASH_E_CUDA;
}

}  // namespace

bool attention_cluster_supported(const AttnArgs& a) {
  const int G = a.nq / a.nkv;
  return a.d == kD && (G == 1 || G == 2 || G == 4 || G == 5 || G == 8);
}

namespace {
// One way to cut a kv head's G query heads over HS clusters of GH heads
// each, with CS CTAs a cluster.
struct Split {
  void (*kern)(ClusterAttnArgs);
  int GH, HS, CS;
};

// The 8-way splits of a group of G, most parallel first.
int splits_for(int G, Split* out) {
  using K = void (*)(ClusterAttnArgs);
  int n = 0;
  auto add = [&](K k, int gh) { out[n++] = Split{k, gh, G / gh, kClusterCtas}; };
  switch (G) {
    case 1: add(attn_cluster_kernel<1, 1, 8>, 1); break;
    case 2: add(attn_cluster_kernel<1, 2, 8>, 1); break;
    case 4: add(attn_cluster_kernel<1, 4, 8>, 1); add(attn_cluster_kernel<2, 2, 8>, 2); break;
    case 5: add(attn_cluster_kernel<1, 5, 8>, 1); add(attn_cluster_kernel<5, 1, 8>, 5); break;
    case 8: add(attn_cluster_kernel<1, 8, 8>, 1); add(attn_cluster_kernel<2, 4, 8>, 2); add(attn_cluster_kernel<4, 2, 8>, 4); break;
    default: break;
  }
  return n;
}

// Many streams: the least split grouping with 2, 4 or 8 CTAs a cluster, in
// that order.
int wide_splits_for(int G, Split* out) {
  int n = 0;
  auto add3 = [&](int gh, auto k2, auto k4, auto k8) {
    out[n++] = Split{k2, gh, G / gh, 2};
    out[n++] = Split{k4, gh, G / gh, 4};
    out[n++] = Split{k8, gh, G / gh, 8};
  };
  switch (G) {
    case 1: add3(1, attn_cluster_kernel<1, 1, 2>, attn_cluster_kernel<1, 1, 4>, attn_cluster_kernel<1, 1, 8>); break;
    case 2: add3(1, attn_cluster_kernel<1, 2, 2>, attn_cluster_kernel<1, 2, 4>, attn_cluster_kernel<1, 2, 8>); break;
    case 4: add3(2, attn_cluster_kernel<2, 2, 2>, attn_cluster_kernel<2, 2, 4>, attn_cluster_kernel<2, 2, 8>); break;
    case 5: add3(5, attn_cluster_kernel<5, 1, 2>, attn_cluster_kernel<5, 1, 4>, attn_cluster_kernel<5, 1, 8>); break;
    case 8: add3(4, attn_cluster_kernel<4, 2, 2>, attn_cluster_kernel<4, 2, 4>, attn_cluster_kernel<4, 2, 8>); break;
    default: break;
  }
  return n;
}

constexpr int kSmemLaunch = ClusterAttnSmem::kBytes + 1024;

// Clusters (of cs CTAs) of this kernel that can be resident at once on this
// device (queried once per kernel; 0 if the query fails).
int resident_clusters(void (*kern)(ClusterAttnArgs), int threads, int cs) {
  static std::mutex mu;
  static std::vector<std::pair<void (*)(ClusterAttnArgs), int>> memo;
  std::lock_guard<std::mutex> lk(mu);
  for (auto& m : memo)
    if (m.first == kern) return m.second;
  int n = 0;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLaunch) == cudaSuccess &&
      cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100) == cudaSuccess) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(cs);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(cs), 1, 1);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = kSmemLaunch;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
  }
  cudaGetLastError();
  memo.emplace_back(kern, n);
  return n;
}
}  // namespace

int attention_cluster_maps(CUtensorMap* kmap, CUtensorMap* vmap, const void* kc, const void* vc, int slabs, int cap) {
  const cuuint64_t dims[3] = {kD, static_cast<cuuint64_t>(cap), static_cast<cuuint64_t>(slabs)};
  const cuuint64_t strides[2] = {kD * 2, static_cast<cuuint64_t>(cap) * kD * 2};
  const cuuint32_t box[3] = {64, kKeys, 1};
  int rc = encode_map(kmap, kc, 3, dims, strides, box);
  if (!rc) rc = encode_map(vmap, vc, 3, dims, strides, box);
  return rc;
}

int launch_attention_cluster(const AttnArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap, int s_count,
                             cudaStream_t st) {
  static thread_local ClusterAttnArgs P;
  P.a = a;
  P.kmap = kmap;
  P.vmap = vmap;
  const int T = s_count * 16;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(a.nkv) * kD, static_cast<cuuint64_t>(T)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(a.nkv) * kD * 2};
  const cuuint32_t box[2] = {64, 16};
  int rc = encode_map(&P.kbmap, a.Kb, 2, dims, strides, box);
  if (!rc) rc = encode_map(&P.vbmap, a.Vb, 2, dims, strides, box);
  if (rc) return rc;
  // Up to four streams: the most parallel 8-way split whose clusters are all
  // resident at once, else the least parallel one; grouping query heads
  // differently gives the same results. More streams: several waves anyway,
  // so the fewest CTAs a cluster that still leave two waves of CTAs (each
  // CTA then carries more keys over its fixed start and reduce costs).
  const int G = a.nq / a.nkv;
  Split sp[4];
  int ns = splits_for(G, sp);
  if (ns == 0) return DFLASH_E_SHAPE;
  int pick = ns - 1;
  if (s_count <= 4) {
    for (int i = 0; i < ns; ++i) {
      const int cap = resident_clusters(sp[i].kern, 32 * (2 * sp[i].GH + 1), sp[i].CS);
      if (cap > 0 && a.nkv * sp[i].HS * s_count <= cap) {
        pick = i;
        break;
      }
    }
  } else {
    ns = wide_splits_for(G, sp);
    if (ns == 0) return DFLASH_E_SHAPE;
    pick = ns - 1;
    for (int i = 0; i < ns; ++i) {
      const int resident_ctas = resident_clusters(sp[i].kern, 32 * (2 * sp[i].GH + 1), sp[i].CS) * sp[i].CS;
      if (resident_ctas > 0 && a.nkv * sp[i].HS * s_count * sp[i].CS >= 2 * resident_ctas) {
        pick = i;
        break;
      }
    }
  }
  void (*kern)(ClusterAttnArgs) = sp[pick].kern;
  const int HS = sp[pick].HS, GH = sp[pick].GH, CS = sp[pick].CS;
  const int threads = 32 * (2 * GH + 1);
  if (resident_clusters(kern, threads, CS) == 0) return DFLASH_E_CUDA;  // also sets the smem attributes
  const int smem = kSmemLaunch;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(CS);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(CS), a.nkv * HS, s_count);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  TraceScope ts(st, "attention", a.trace_bytes, 0.0);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, P);
  count_launch();
  return cuda_status(e);
}

}  // namespace dfl
