// Non-causal block attention of the drafter: the 16 block rows of a stream
// attend the layer's visible context (full layer: every committed position;
// sliding layer: the ring of its last W positions) plus the block's own 16
// rows, with grouped-query heads.
//
// Work unit = (chunk of context slots, kv head, stream). The group of query
// heads that share the kv head (4 for 32/8 heads) is one warp each, 16 query
// rows per warp, so one K/V tile staged in shared memory serves the whole
// group. Scores and P*V run on the tensor cores (mma.sync m16n8k16 bf16,
// fp32 accumulate; P enters as a bf16 hi + lo pair so P*V keeps fp32-level
// accuracy) with an online softmax; chunk 0 also covers the block's
// 16 rows. Each unit writes its unnormalised output and (max, sum); a second
// kernel merges the chunks with their log-sum-exp weights. Chunk sizes depend
// only on the layer's cache capacity, so a stream's result does not depend on
// the other streams in the batch.
#include "internal.h"
#include "ptx.cuh"

namespace dfl {

namespace {

constexpr int kKeysPerTile = 64;

__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], uint32_t saddr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(saddr));
}

__device__ __forceinline__ void cp_async16(uint32_t saddr, const void* g, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(saddr), "l"(g), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// (a, b) -> bf16 pairs hi = bf16(x), lo = bf16(x - hi)
__device__ __forceinline__ void split_bf16(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  const float2 hf = __bfloat1622float2(h);
  const __nv_bfloat162 l = __floats2bfloat162_rn(a - hf.x, b - hf.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

template <int D>
struct AttnSmem {
  static constexpr int kLd = D + 8;  // padded row (bf16) so fragment loads hit distinct banks
  static constexpr int kTileElems = kKeysPerTile * kLd;
  static constexpr int kBytes = 2 /*buffers*/ * 2 /*K,V*/ * kTileElems * 2;
};

// Source row of key `k` of a unit: context slots first, then the block rows.
template <int D>
__device__ __forceinline__ const __nv_bfloat16* key_row(const __nv_bfloat16* cache, const __nv_bfloat16* blk, int k,
                                                        int nctx, int r0, int64_t cache_base, int64_t blk_base,
                                                        int blk_ld) {
  if (k < nctx) return cache + cache_base + static_cast<int64_t>(r0 + k) * D;
  return blk + blk_base + static_cast<int64_t>(k - nctx) * blk_ld;
}

template <int D>
__device__ __forceinline__ void load_tile(__nv_bfloat16* Ks, __nv_bfloat16* Vs, const AttnArgs& a, int tile, int nk,
                                          int nctx, int r0, int64_t cache_base, int64_t blk_base) {
  constexpr int kChunks = D / 8;  // 16-byte pieces per row
  const int blk_ld = a.nkv * D;
  for (int idx = threadIdx.x; idx < kKeysPerTile * kChunks; idx += blockDim.x) {
    const int r = idx / kChunks;
    const int c = idx - r * kChunks;
    const int k = tile * kKeysPerTile + r;
    const bool ok = k < nk;
    const int kk = ok ? k : 0;
    const __nv_bfloat16* gk = key_row<D>(a.Kc, a.Kb, kk, nctx, r0, cache_base, blk_base, blk_ld) + c * 8;
    const __nv_bfloat16* gv = key_row<D>(a.Vc, a.Vb, kk, nctx, r0, cache_base, blk_base, blk_ld) + c * 8;
    const uint32_t sk = static_cast<uint32_t>(__cvta_generic_to_shared(Ks + r * AttnSmem<D>::kLd + c * 8));
    const uint32_t sv = static_cast<uint32_t>(__cvta_generic_to_shared(Vs + r * AttnSmem<D>::kLd + c * 8));
    cp_async16(sk, gk, ok ? 16 : 0);  // rows past the unit are zero-filled
    cp_async16(sv, gv, ok ? 16 : 0);
  }
}

template <int D>
__global__ void __launch_bounds__(256) attn_kernel(const AttnArgs a) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  __nv_bfloat16* buf = reinterpret_cast<__nv_bfloat16*>(smem_raw);
  constexpr int kLd = AttnSmem<D>::kLd;
  constexpr int kTE = AttnSmem<D>::kTileElems;
  pdl_trigger();
  pdl_wait();

  const int c = blockIdx.x;
  const int kvh = blockIdx.y;
  const int si = blockIdx.z;
  const int s = a.s_begin + si;
  const int C = a.lens[s];
  const int nvis = a.window > 0 ? min(C, a.window) : C;
  const int r0 = c * a.chunk;
  if (c > 0 && r0 >= nvis) return;
  const int nctx = max(0, min(r0 + a.chunk, nvis) - r0);
  const int nk = nctx + (c == 0 ? 16 : 0);
  const int ntiles = (nk + kKeysPerTile - 1) / kKeysPerTile;
  const int G = a.nq / a.nkv;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int h = kvh * G + warp;
  const int64_t cache_base = (static_cast<int64_t>(s) * a.nkv + kvh) * a.cap * D;
  const int64_t blk_base = static_cast<int64_t>(si) * 16 * (a.nkv * D) + kvh * D;

  // Q fragments (A operand, row-major 16 x D) straight from global memory
  uint32_t qa[D / 16][4];
  {
    const __nv_bfloat16* Q = a.Q + static_cast<int64_t>(si) * 16 * (a.nq * D) + static_cast<int64_t>(h) * D;
    const int qr = lane >> 2;
    const int qc = (lane & 3) * 2;
    const int ld = a.nq * D;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      qa[kk][0] = *reinterpret_cast<const uint32_t*>(Q + qr * ld + kk * 16 + qc);
      qa[kk][1] = *reinterpret_cast<const uint32_t*>(Q + (qr + 8) * ld + kk * 16 + qc);
      qa[kk][2] = *reinterpret_cast<const uint32_t*>(Q + qr * ld + kk * 16 + qc + 8);
      qa[kk][3] = *reinterpret_cast<const uint32_t*>(Q + (qr + 8) * ld + kk * 16 + qc + 8);
    }
  }

  float o[D / 8][4];
#pragma unroll
  for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float mrow[2] = {-INFINITY, -INFINITY};
  float lrow[2] = {0.f, 0.f};
  const float sc = rsqrtf(static_cast<float>(D)) * 1.4426950408889634f;  // 1/sqrt(d) * log2(e)

  load_tile<D>(buf, buf + kTE, a, 0, nk, nctx, r0, cache_base, blk_base);
  cp_async_commit();
  for (int t = 0; t < ntiles; ++t) {
    const int cur = t & 1;
    if (t + 1 < ntiles) {
      load_tile<D>(buf + (cur ^ 1) * 2 * kTE, buf + (cur ^ 1) * 2 * kTE + kTE, a, t + 1, nk, nctx, r0, cache_base,
                   blk_base);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    if (warp < G) {
      const __nv_bfloat16* Ks = buf + cur * 2 * kTE;
      const __nv_bfloat16* Vs = Ks + kTE;
      // S = Q K^T for 64 keys: 8 n-tiles of 8 keys
      float sacc[8][4];
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        sacc[n][0] = sacc[n][1] = sacc[n][2] = sacc[n][3] = 0.f;
        const __nv_bfloat16* kr = Ks + (n * 8 + (lane >> 2)) * kLd + (lane & 3) * 2;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t b0 = *reinterpret_cast<const uint32_t*>(kr + kk * 16);
          const uint32_t b1 = *reinterpret_cast<const uint32_t*>(kr + kk * 16 + 8);
          mma_bf16_16816(sacc[n], qa[kk], b0, b1);
        }
      }
      // online softmax (rows lane/4 and lane/4 + 8)
      const int kbase = t * kKeysPerTile;
      float tmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int n = 0; n < 8; ++n) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int key = kbase + n * 8 + (lane & 3) * 2 + (e & 1);
          const float v = key < nk ? sacc[n][e] * sc : -INFINITY;
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
        mnew[r] = fmaxf(mrow[r], tmax[r]);
        alpha[r] = exp2f(mrow[r] - mnew[r]);  // exp2(-inf) = 0 on the first tile
        mrow[r] = mnew[r];
      }
#pragma unroll
      for (int n = 0; n < 8; ++n) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float p = exp2f(sacc[n][e] - mnew[e >> 1]);
          sacc[n][e] = p;
          psum[e >> 1] += p;
        }
      }
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        psum[r] += __shfl_xor_sync(0xffffffffu, psum[r], 1);
        psum[r] += __shfl_xor_sync(0xffffffffu, psum[r], 2);
        lrow[r] = lrow[r] * alpha[r] + psum[r];
      }
#pragma unroll
      for (int n = 0; n < D / 8; ++n) {
        o[n][0] *= alpha[0];
        o[n][1] *= alpha[0];
        o[n][2] *= alpha[1];
        o[n][3] *= alpha[1];
      }
      // O += P V with P split into bf16 hi + lo parts (P = hi + lo to ~2^-17),
      // so the product keeps fp32-level accuracy; V via transposed ldmatrix
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        uint32_t ph[4], pl[4];
        split_bf16(sacc[2 * kk][0], sacc[2 * kk][1], ph[0], pl[0]);
        split_bf16(sacc[2 * kk][2], sacc[2 * kk][3], ph[1], pl[1]);
        split_bf16(sacc[2 * kk + 1][0], sacc[2 * kk + 1][1], ph[2], pl[2]);
        split_bf16(sacc[2 * kk + 1][2], sacc[2 * kk + 1][3], ph[3], pl[3]);
        const int mi = lane >> 3;
        const int key = kk * 16 + (mi & 1) * 8 + (lane & 7);
#pragma unroll
        for (int n2 = 0; n2 < D / 16; ++n2) {
          const int dim = n2 * 16 + (mi >> 1) * 8;
          uint32_t vb[4];
          ldmatrix_x4_trans(vb, static_cast<uint32_t>(__cvta_generic_to_shared(Vs + key * kLd + dim)));
          mma_bf16_16816(o[2 * n2], ph, vb[0], vb[1]);
          mma_bf16_16816(o[2 * n2 + 1], ph, vb[2], vb[3]);
          mma_bf16_16816(o[2 * n2], pl, vb[0], vb[1]);
          mma_bf16_16816(o[2 * n2 + 1], pl, vb[2], vb[3]);
        }
      }
    }
    __syncthreads();  // the buffer is refilled next iteration
  }

  if (warp < G) {
    const size_t unit = (static_cast<size_t>(si) * a.nq + h) * a.nchunk + c;
    float* po = a.part_o + unit * 16 * D;
    float* pml = a.part_ml + unit * 16 * 2;
    const int r = lane >> 2;
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      const int col = n * 8 + (lane & 3) * 2;
      *reinterpret_cast<float2*>(po + r * D + col) = make_float2(o[n][0], o[n][1]);
      *reinterpret_cast<float2*>(po + (r + 8) * D + col) = make_float2(o[n][2], o[n][3]);
    }
    if ((lane & 3) == 0) {
      pml[r * 2] = mrow[0];
      pml[r * 2 + 1] = lrow[0];
      pml[(r + 8) * 2] = mrow[1];
      pml[(r + 8) * 2 + 1] = lrow[1];
    }
  }
}

// Merge the chunks of one (stream, query head, row): O = sum_c 2^(m_c - M) O_c
// / sum_c 2^(m_c - M) l_c, in chunk order. One warp per output row vector,
// each lane owning D/32 consecutive dims.
template <int D>
__global__ void __launch_bounds__(256) attn_combine_kernel(const AttnArgs a, int s_count) {
  pdl_trigger();
  pdl_wait();
  constexpr int kPer = D / 32;
  const int wg = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (wg >= s_count * a.nq * 16) return;
  const int r = wg & 15;
  const int h = (wg >> 4) % a.nq;
  const int si = (wg >> 4) / a.nq;
  const int s = a.s_begin + si;
  const int C = a.lens[s];
  const int nvis = a.window > 0 ? min(C, a.window) : C;
  const int nu = max(1, (nvis + a.chunk - 1) / a.chunk);
  const size_t unit0 = (static_cast<size_t>(si) * a.nq + h) * a.nchunk;
  const float* ml = a.part_ml + unit0 * 32 + r * 2;
  float M = -INFINITY;
  for (int u = lane; u < nu; u += 32) M = fmaxf(M, ml[u * 32]);
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  float acc[kPer];
#pragma unroll
  for (int p = 0; p < kPer; ++p) acc[p] = 0.f;
  float den = 0.f;
  const float* po = a.part_o + (unit0 * 16 + r) * D + lane * kPer;
#pragma unroll 4
  for (int u = 0; u < nu; ++u) {
    const float w = exp2f(ml[u * 32] - M);
    den += w * ml[u * 32 + 1];
    const float* pu = po + static_cast<size_t>(u) * 16 * D;
    if constexpr (kPer == 4) {
      const float4 v = *reinterpret_cast<const float4*>(pu);
      acc[0] += w * v.x;
      acc[1] += w * v.y;
      acc[2] += w * v.z;
      acc[3] += w * v.w;
    } else {
#pragma unroll
      for (int p = 0; p < kPer; ++p) acc[p] += w * pu[p];
    }
  }
  __nv_bfloat16* out = a.out + (static_cast<int64_t>(si) * 16 + r) * (a.nq * D) + h * D + lane * kPer;
#pragma unroll
  for (int p = 0; p < kPer; ++p) out[p] = __float2bfloat16_rn(acc[p] / den);
}

template <int D>
int launch_d(const AttnArgs& a, int s_count, cudaStream_t st) {
  const int G = a.nq / a.nkv;
  const int smem = AttnSmem<D>::kBytes;
  static bool configured = false;
  if (!configured) {
    if (cudaFuncSetAttribute(attn_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return DFLASH_E_CUDA;
    configured = true;
  }
  dim3 grid(a.nchunk, a.nkv, s_count);
  {
    TraceScope ts(st, "attention", a.trace_bytes, 0.0);
    const cudaError_t e = launch_pdl(attn_kernel<D>, grid, dim3(32 * G), smem, st, a);
    count_launch();
    if (e != cudaSuccess) return DFLASH_E_CUDA;
  }
  const int warps = s_count * a.nq * 16;
  dim3 g2((warps + 7) / 8);
  {
    TraceScope ts(st, "attention.combine", static_cast<double>(s_count) * a.nq * 16 * D * 2, 0.0);
    const cudaError_t e = launch_pdl(attn_combine_kernel<D>, g2, dim3(256), 0, st, a, s_count);
    count_launch();
    if (e != cudaSuccess) return DFLASH_E_CUDA;
  }
  return cuda_status(cudaGetLastError());
}

}  // namespace

size_t attn_partial_floats(int s_count, int nq, int nchunk, int d) {
  return static_cast<size_t>(s_count) * nq * nchunk * 16 * (d + 2);
}

int launch_attention(const AttnArgs& a, int s_count, cudaStream_t st) {
  const int G = a.nq / a.nkv;
  if (G < 1 || G > 8) return DFLASH_E_SHAPE;
  switch (a.d) {
    case 32:
      return launch_d<32>(a, s_count, st);
    case 64:
      return launch_d<64>(a, s_count, st);
    case 128:
      return launch_d<128>(a, s_count, st);
    default:
      return DFLASH_E_SHAPE;
  }
}

}  // namespace dfl
