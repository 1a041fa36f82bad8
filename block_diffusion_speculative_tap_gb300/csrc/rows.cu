// Row-wise kernels of the hot path: block embedding, RMSNorm of the fp32
// residual into bf16 GEMM operands, the hidden_norm that turns fc's output
// into fused ring rows, the K/V rows of wide fills, and the bookkeeping of
// appended rows.
//
// A row's sum of squares arrives as per-128-feature parts (published by the
// kernel that wrote the row, or by row_sumsq) and is summed in one fixed
// order, so the norms are elementwise and a row's result does not depend on
// which other rows share the launch.
#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

namespace dfl {

namespace {

// Per-128-feature sums of squares of one row, ss[p * ss_ld + t], for an
// input norm fused into the GEMM that reads the row next (lane sums of four
// in order, then a fixed warp tree). Warp w of the CTA takes parts w, w + 4,
// ...; `x4(i)` yields float4 i of the row.
constexpr int kStatThreads = 128;

template <typename Load>
__device__ __forceinline__ void row_sumsq(float* __restrict__ ss, int ss_ld, int t, int H, Load x4) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int p = warp; p * 128 < H; p += kStatThreads / 32) {
    const float4 v = x4(p * 32 + lane);
    float q = ((v.x * v.x + v.y * v.y) + v.z * v.z) + v.w * v.w;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) q += __shfl_xor_sync(0xffffffffu, q, off);
    if (lane == 0) ss[static_cast<int64_t>(p) * ss_ld + t] = q;
  }
}

// rstd of row r from its per-128-feature sums of squares ss[p][r]: lane l
// adds parts l, l + 32, ... in order, then a fixed xor butterfly over the
// lanes (five steps instead of a 32-step chain; floating-point addition is
// commutative, so every lane ends with the same value, and the order is the
// same for every row and launch).
__device__ __forceinline__ float parts_rstd(const float* __restrict__ ss, int ss_ld, int r, int H, float inv_h,
                                            float eps) {
  const int lane = threadIdx.x & 31;
  const int parts = H / 128;
  float sum = 0.f;
  for (int p = lane; p < parts; p += 32) sum += __ldcg(&ss[static_cast<int64_t>(p) * ss_ld + r]);
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  return rsqrtf(__fmaf_rn(sum, inv_h, eps));
}

// X[t] = embed[token_t] as fp32; token 16s is the anchor of stream s, the
// other fifteen rows of the block are the mask token [anchor + 15 mask rows].
// The row's sums of squares go to ss, and (xn != null) its RMSNorm with gain
// g to xn, with the arithmetic of rmsnorm_rows_kernel (the first layer's
// input norm needs no launch of its own).
__global__ void __launch_bounds__(kStatThreads) embed_kernel(float* __restrict__ X, float* __restrict__ ss,
                                                             const __nv_bfloat16* __restrict__ E,
                                                             const int* __restrict__ anchors, int H, int V, int mask,
                                                             int ss_ld, int* err, int* __restrict__ zero, int nzero,
                                                             __nv_bfloat16* __restrict__ xn,
                                                             const __nv_bfloat16* __restrict__ g, float inv_h,
                                                             float eps) {
  pdl_trigger();
  pdl_wait();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < nzero; i += gridDim.x * blockDim.x) zero[i] = 0;
  const int t = blockIdx.x;
  int tok = mask;
  if ((t & 15) == 0) {
    tok = anchors[t >> 4];
    if (tok < 0 || tok >= V) {
      if (threadIdx.x == 0) atomicOr(err, DFLASH_STATUS_BAD_TOKEN);
      tok = 0;
    }
  }
  const uint2* e = reinterpret_cast<const uint2*>(E + static_cast<int64_t>(tok) * H);
  float4* x = reinterpret_cast<float4*>(X + static_cast<int64_t>(t) * H);
  row_sumsq(ss, ss_ld, t, H, [&](int i) {
    const uint2 r = e[i];
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r.y));
    const float4 v = make_float4(a.x, a.y, b.x, b.y);
    x[i] = v;
    return v;
  });
  if (xn == nullptr) return;
  __syncthreads();  // the row's part sums and values are written
  const float rstd = parts_rstd(ss, ss_ld, t, H, inv_h, eps);
  for (int i = threadIdx.x; i < H / 8; i += blockDim.x) {
    const float4 a = x[2 * i], b = x[2 * i + 1];
    const uint4 gr = *reinterpret_cast<const uint4*>(g + 8 * i);
    const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&gr);
    const float xs[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint4 o;
    uint32_t* o2 = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 gf = __bfloat1622float2(g2[k]);
      const __nv_bfloat162 y = __floats2bfloat162_rn(xs[2 * k] * rstd * gf.x, xs[2 * k + 1] * rstd * gf.y);
      o2[k] = *reinterpret_cast<const uint32_t*>(&y);
    }
    *reinterpret_cast<uint4*>(xn + static_cast<int64_t>(t) * H + 8 * i) = o;
  }
}

// Sums of squares of rows of a caller-given residual X.
__global__ void __launch_bounds__(kStatThreads) row_sumsq_kernel(float* __restrict__ ss, const float* __restrict__ X,
                                                                 int H, int ss_ld) {
  pdl_trigger();
  pdl_wait();
  const int t = blockIdx.x;
  const float4* x = reinterpret_cast<const float4*>(X + static_cast<int64_t>(t) * H);
  row_sumsq(ss, ss_ld, t, H, [&](int i) { return x[i]; });
}

// out[r] = bf16(x[src] * rstd * g), rstd = 1 / sqrt(sum_p ss[p][src] / H +
// eps): the row's sum of squares comes as per-128-feature parts published by
// the kernel that wrote the row (summed here in one fixed order), so the norm is
// elementwise. A CTA covers 1024 features of one row, 8 a thread.
constexpr int kNormThreads = 128;

__global__ void __launch_bounds__(kNormThreads) rmsnorm_rows_kernel(__nv_bfloat16* __restrict__ out,
                                                                    const float* __restrict__ x,
                                                                    const __nv_bfloat16* __restrict__ g,
                                                                    const float* __restrict__ ss, int ss_ld, int H,
                                                                    float inv_h, float eps, int mask_rows_only) {
  pdl_trigger();
  const int r = blockIdx.y;
  const int src = mask_rows_only ? (r / 15) * 16 + 1 + (r % 15) : r;
  const int i = (blockIdx.x * kNormThreads + threadIdx.x) * 8;  // first feature
  const bool live = i < H;
  // the gain is a weight: loaded before the wait; the row's values are
  // loaded before its sum of squares is reduced (no round trip in between)
  const uint4 gr = live ? *reinterpret_cast<const uint4*>(g + i) : make_uint4(0, 0, 0, 0);
  pdl_wait();
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
  if (live) {
    const float4* xr = reinterpret_cast<const float4*>(x + static_cast<int64_t>(src) * H + i);
    a = __ldcg(xr);
    b = __ldcg(xr + 1);
  }
  const float rstd = parts_rstd(ss, ss_ld, src, H, inv_h, eps);
  if (!live) return;
  const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&gr);
  const float xs[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  uint4 o;
  uint32_t* o2 = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 gf = __bfloat1622float2(g2[k]);
    const __nv_bfloat162 y = __floats2bfloat162_rn(xs[2 * k] * rstd * gf.x, xs[2 * k + 1] * rstd * gf.y);
    o2[k] = *reinterpret_cast<const uint32_t*>(&y);
  }
  *reinterpret_cast<uint4*>(out + static_cast<int64_t>(r) * H + i) = o;
}

// fused = bf16(RMSNorm(y) * hidden_norm), rstd from the sums of squares the
// fc GEMM published: written to the ring slot of the row's (stream,
// position) and to a dense staging copy for K/V injection. Elementwise: a CTA
// covers 1024 features of one row, 8 a thread.
__global__ void __launch_bounds__(128) hidden_norm_kernel(__nv_bfloat16* __restrict__ ring,
                                                          __nv_bfloat16* __restrict__ fused_tmp,
                                                          const float* __restrict__ y, const float* __restrict__ ss,
                                                          const __nv_bfloat16* __restrict__ g,
                                                          const int* __restrict__ row_stream,
                                                          const int* __restrict__ row_pos, int rows, int H, int R,
                                                          float inv_h, float eps) {
  pdl_trigger();
  pdl_wait();
  const int r = blockIdx.y;
  const int i = (blockIdx.x * 128 + threadIdx.x) * 8;
  const bool live = i < H;
  // the row's values are loaded before its sum of squares is reduced
  const uint4 gr = live ? *reinterpret_cast<const uint4*>(g + i) : make_uint4(0, 0, 0, 0);
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
  if (live) {
    const float4* yr = reinterpret_cast<const float4*>(y + static_cast<int64_t>(r) * H + i);
    a = __ldcg(yr);
    b = __ldcg(yr + 1);
  }
  const float rstd = parts_rstd(ss, rows, r, H, inv_h, eps);
  if (!live) return;
  const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&gr);
  const float xs[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  uint4 o;
  uint32_t* o2 = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 gf = __bfloat1622float2(g2[k]);
    const __nv_bfloat162 v = __floats2bfloat162_rn(xs[2 * k] * rstd * gf.x, xs[2 * k + 1] * rstd * gf.y);
    o2[k] = *reinterpret_cast<const uint32_t*>(&v);
  }
  *reinterpret_cast<uint4*>(ring + (static_cast<int64_t>(row_stream[r]) * R + row_pos[r]) * H + i) = o;
  *reinterpret_cast<uint4*>(fused_tmp + static_cast<int64_t>(r) * H + i) = o;
}

// K/V injection of wide fills, second half: the GEMM left the raw
// projections y [rows][ld] (fp32, all segments side by side); one warp per
// (row, head) applies k_norm (K segments: per-head RMSNorm over d, gain) and
// rotate-half RoPE at the row's position, and stores bf16 to the head's cache
// slot. Lane l holds features q*32 + l, q < d/32; the sum of squares of a
// head is a xor tree per q and then the q's in order, the same arithmetic
// as the fused epilogue.
__global__ void __launch_bounds__(256) kv_rows_kernel(const float* __restrict__ y, int64_t ld, const KvSegs segs,
                                                      const int* __restrict__ row_stream,
                                                      const int* __restrict__ row_pos,
                                                      const int* __restrict__ row_end,
                                                      const float2* __restrict__ rope, int d, float eps, int rows) {
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x;
  const int hh = blockIdx.y * 8 + (threadIdx.x >> 5);  // head over all segments
  if (r >= rows || hh >= segs.head0[segs.n]) return;
  int s = 0;
  while (s + 1 < segs.n && hh >= segs.head0[s + 1]) ++s;
  const int head = hh - segs.head0[s];
  const int pos = row_pos[r];
  const int window = segs.window[s];
  if (window > 0 && pos < row_end[r] - window) return;  // a later row of the segment owns this ring slot
  const int nq = d >> 5;
  const float* src = y + static_cast<int64_t>(r) * ld + segs.col0[s] + static_cast<int64_t>(head) * d;
  float v[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) v[q] = q < nq ? src[q * 32 + lane] : 0.f;
  if (segs.gain[s] != nullptr) {
    float tot = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (q < nq) {
        float t = v[q] * v[q];
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
        tot = q == 0 ? t : tot + t;
      }
    }
    const float inv_d = 1.0f / static_cast<float>(d);  // d is a power of two: exact
    const float rs = head_norm_scale(tot, inv_d, eps);
    const int half = d >> 1;
    float yv[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (q < nq) {
        const int dim = q * 32 + lane;
        yv[q] = head_norm_apply(v[q], rs, __bfloat162float(segs.gain[s][dim]));
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (q < nq) {
        const int dim = q * 32 + lane;
        const int fi = dim < half ? dim : dim - half;
        // the partner feature dim +- d/2: another q of this lane, or lane ^ 16 when d = 32
        float yp;
        if (nq == 1)
          yp = __shfl_xor_sync(0xffffffffu, yv[0], 16);
        else
          yp = yv[q ^ (nq >> 1)];
        const float2 cs = rope[static_cast<int64_t>(pos) * half + fi];
        v[q] = rope_rotate(yv[q], yp, cs, dim < half);
      }
    }
  }
  const int slot = window > 0 ? pos % window : pos;
  __nv_bfloat16* dst =
      segs.dst[s] + ((static_cast<int64_t>(row_stream[r]) * segs.heads[s] + head) * segs.cap[s] + slot) * d;
#pragma unroll
  for (int q = 0; q < 4; ++q)
    if (q < nq) dst[q * 32 + lane] = __float2bfloat16_rn(v[q]);
}

struct SegTable {
  int n;
  int stream[256];
  int start[256];
  int rows[256];
  int first_row[257];
};

// Row tables of the appended rows, the new stream lengths (lens != null) and
// a zeroed range of split-K counters (kernel-side, so the launch sequence has
// no memset node to break the programmatic-dependent-launch chain).
__global__ void prep_rows_kernel(int* __restrict__ row_stream, int* __restrict__ row_pos, int* __restrict__ row_end,
                                 const SegTable tab, int total, int* __restrict__ lens, int* __restrict__ zero,
                                 int nzero) {
  pdl_trigger();
  pdl_wait();
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  for (int i = r; i < nzero; i += gridDim.x * blockDim.x) zero[i] = 0;
  if (lens != nullptr && r < tab.n) lens[tab.stream[r]] = tab.start[r] + tab.rows[r];
  if (r >= total) return;
  int s = 0;
  while (s + 1 < tab.n && r >= tab.first_row[s + 1]) ++s;
  row_stream[r] = tab.stream[s];
  row_pos[r] = tab.start[s] + (r - tab.first_row[s]);
  row_end[r] = tab.start[s] + tab.rows[s];
}

// A bounded wait on an mbarrier that nothing arrives at: it gives up after
// `limit` cycles and sets the timeout bit of *err, as any expired wait of the
// hot path does (the self-test of that mechanism).
__global__ void wait_probe_kernel(int* err, long long limit) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
    mbar_wait(&bar, 0, err, DFLASH_STATUS_TIMEOUT, nullptr, limit);
  }
}

}  // namespace

int launch_wait_probe(int* err, long long cycles, cudaStream_t st) {
  wait_probe_kernel<<<1, 32, 0, st>>>(err, cycles);
  count_launch();
  return cuda_status(cudaGetLastError());
}

namespace {

// ---------------------------------------------------------------- two-tap dynamic convolution
// DFlash2's dynamic short convolution over the block's rows: from the normed
// rows h = bf16(RMSNorm(X) * conv_norm), the tap logits z[t] = h[t] . proj^T
// (2 * groups of them a row), then X[t] += a0 * h[t - 1] + a1 * h[t] with
// (a0, a1) = softmax(z[t][2g], z[t][2g + 1]) for the channel's group g.
constexpr int kConvThreads = 256;

// A warp a logit: lanes take 8-feature pieces in order, then a fixed xor tree.
__global__ void __launch_bounds__(kConvThreads) conv_logits_kernel(const __nv_bfloat16* __restrict__ h,
                                                                   const __nv_bfloat16* __restrict__ proj, int H,
                                                                   int nz, float* __restrict__ z) {
  pdl_trigger();
  pdl_wait();
  const int t = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint4* hr = reinterpret_cast<const uint4*>(h + static_cast<int64_t>(t) * H);
  for (int q = warp; q < nz; q += kConvThreads / 32) {
    const uint4* pr = reinterpret_cast<const uint4*>(proj + static_cast<int64_t>(q) * H);
    float acc = 0.f;
    for (int i = lane; i < H / 8; i += 32) {
      const uint4 a = hr[i], b = __ldg(pr + i);
      const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
      const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 fa = __bfloat1622float2(a2[k]), fb = __bfloat1622float2(b2[k]);
        acc = fmaf(fa.x, fb.x, acc);
        acc = fmaf(fa.y, fb.y, acc);
      }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) z[static_cast<int64_t>(t) * nz + q] = acc;
  }
}

// Elementwise mix: a CTA covers 1024 features of one row, 8 a thread (one
// group: a group holds a multiple of 16 features); a stream's first row (the
// anchor's) has no row before it.
__global__ void __launch_bounds__(128) conv_mix_kernel(float* __restrict__ X, const __nv_bfloat16* __restrict__ h,
                                                       const float* __restrict__ z, int H, int groups) {
  pdl_trigger();
  pdl_wait();
  const int t = blockIdx.y;
  const int i = (blockIdx.x * 128 + threadIdx.x) * 8;
  if (i >= H) return;
  const int g = i / (H / groups);
  const float z0 = z[static_cast<int64_t>(t) * 2 * groups + 2 * g];
  const float z1 = z[static_cast<int64_t>(t) * 2 * groups + 2 * g + 1];
  const float m = fmaxf(z0, z1);
  const float e0 = expf(z0 - m), e1 = expf(z1 - m);
  const float inv = 1.f / (e0 + e1);
  const float a0 = e0 * inv, a1 = e1 * inv;
  const uint4 hc = *reinterpret_cast<const uint4*>(h + static_cast<int64_t>(t) * H + i);
  const uint4 hp = (t & 15) ? *reinterpret_cast<const uint4*>(h + static_cast<int64_t>(t - 1) * H + i)
                            : make_uint4(0u, 0u, 0u, 0u);
  const __nv_bfloat162* c2 = reinterpret_cast<const __nv_bfloat162*>(&hc);
  const __nv_bfloat162* p2 = reinterpret_cast<const __nv_bfloat162*>(&hp);
  float4* xr = reinterpret_cast<float4*>(X + static_cast<int64_t>(t) * H + i);
  float4 x0 = xr[0], x1 = xr[1];
  float* xs[8] = {&x0.x, &x0.y, &x0.z, &x0.w, &x1.x, &x1.y, &x1.z, &x1.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 fc = __bfloat1622float2(c2[k]), fp = __bfloat1622float2(p2[k]);
    *xs[2 * k] += a0 * fp.x + a1 * fc.x;
    *xs[2 * k + 1] += a0 * fp.y + a1 * fc.y;
  }
  xr[0] = x0;
  xr[1] = x1;
}

}  // namespace

int launch_block_conv(float* X, const __nv_bfloat16* h, float* z, const __nv_bfloat16* proj, int S, int H, int groups,
                      cudaStream_t st) {
  if (S <= 0) return DFLASH_OK;
  if (groups < 1 || groups > kMaxConvGroups || H % groups || (H / groups) % 16) return DFLASH_E_SHAPE;
  const int T = S * DFLASH_BLOCK, nz = 2 * groups;
  {
    TraceScope ts(st, "conv.taps", static_cast<double>(T) * H * 2 + static_cast<double>(nz) * H * 2 + T * nz * 4.0,
                  2.0 * T * nz * H);
    const cudaError_t e = launch_pdl(conv_logits_kernel, dim3(T), dim3(kConvThreads), 0, st, h, proj, H, nz, z);
    count_launch();
    if (e != cudaSuccess) return DFLASH_E_CUDA;
  }
  TraceScope ts(st, "conv.mix", static_cast<double>(T) * H * 10 + T * nz * 4.0, 0.0);
  const cudaError_t e =
      launch_pdl(conv_mix_kernel, dim3((H + 1023) / 1024, T), dim3(128), 0, st, X, h, static_cast<const float*>(z), H, groups);
  count_launch();
  return cuda_status(e);
}

int launch_embed(float* X, float* ss, const __nv_bfloat16* embed, const int* anchors, int S, int H, int V, int mask,
                 int* err, int* zero, int nzero, __nv_bfloat16* xn, const __nv_bfloat16* g, float eps,
                 cudaStream_t st) {
  TraceScope ts(st, "embed", static_cast<double>(S) * 16 * H * 6 + static_cast<double>(S) * 16 * (H / 128) * 4, 0.0);
  // a plain launch: the draft's first kernel starts after all earlier work on
  // the stream (the fills whose K/V rows and lengths the attention of this
  // call reads before its own programmatic-dependence wait) has completed
  embed_kernel<<<dim3(S * 16), dim3(kStatThreads), 0, st>>>(X, ss, embed, anchors, H, V, mask, S * 16, err, zero, nzero,
                                                            xn, g, 1.0f / static_cast<float>(H), eps);
  const cudaError_t e = cudaGetLastError();
  count_launch();
  return cuda_status(e);
}

int launch_row_sumsq(float* ss, const float* X, int rows, int H, cudaStream_t st) {
  TraceScope ts(st, "row_sumsq", static_cast<double>(rows) * H * 4 + static_cast<double>(rows) * (H / 128) * 4, 0.0);
  const cudaError_t e = launch_pdl(row_sumsq_kernel, dim3(rows), dim3(kStatThreads), 0, st, ss, X, H, rows);
  count_launch();
  return cuda_status(e);
}

int launch_rmsnorm_rows(__nv_bfloat16* out, const float* x, const __nv_bfloat16* g, const float* ss, int ss_ld,
                        int rows, int H, float eps, int mask_rows_only, cudaStream_t st) {
  if (H % 8) return DFLASH_E_SHAPE;
  TraceScope ts(st, "rmsnorm", static_cast<double>(rows) * H * 6 + static_cast<double>(rows) * (H / 128) * 4, 0.0);
  const dim3 grid((H + kNormThreads * 8 - 1) / (kNormThreads * 8), rows);
  const cudaError_t e = launch_pdl(rmsnorm_rows_kernel, grid, dim3(kNormThreads), 0, st, out, x, g, ss, ss_ld, H,
                                   1.0f / static_cast<float>(H), eps, mask_rows_only);
  count_launch();
  return cuda_status(e);
}

int launch_kv_rows(const float* y, int64_t ld, const KvSegs& segs, const int* row_stream, const int* row_pos,
                   const int* row_end, const float2* rope, int d, float eps, int rows, cudaStream_t st) {
  if (rows <= 0) return DFLASH_OK;
  if (d != 32 && d != 64 && d != 128) return DFLASH_E_SHAPE;
  const int heads = segs.head0[segs.n];
  TraceScope ts(st, "kv_rows", static_cast<double>(rows) * heads * d * 6.0, 0.0);
  const cudaError_t e = launch_pdl(kv_rows_kernel, dim3(rows, (heads + 7) / 8), dim3(256), 0, st, y, ld, segs,
                                   row_stream, row_pos, row_end, rope, d, eps, rows);
  count_launch();
  return cuda_status(e);
}

int launch_hidden_norm(__nv_bfloat16* ring, __nv_bfloat16* fused_tmp, const float* y, const float* ss,
                       const __nv_bfloat16* g, const int* row_stream, const int* row_pos, int rows, int H, int R,
                       float eps, cudaStream_t st) {
  if (H % 8) return DFLASH_E_SHAPE;
  TraceScope ts(st, "hidden_norm", static_cast<double>(rows) * H * 8, 0.0);
  const dim3 grid((H + 1023) / 1024, rows);
  const cudaError_t e = launch_pdl(hidden_norm_kernel, grid, dim3(128), 0, st, ring, fused_tmp, y, ss, g, row_stream,
                                   row_pos, rows, H, R, 1.0f / static_cast<float>(H), eps);
  count_launch();
  return cuda_status(e);
}

// seg_info_host_packed: 3*nseg ints (stream, start, rows) on the host.
int launch_prep_rows(int* row_stream, int* row_pos, int* row_end, int* lens, int nseg, int rows,
                     const int* seg_info_host_packed, int* zero, int nzero, cudaStream_t st) {
  if (nseg < 1 || nseg > 256) return DFLASH_E_INVALID_ARG;
  SegTable tab{};
  tab.n = nseg;
  tab.first_row[0] = 0;
  for (int i = 0; i < nseg; ++i) {
    tab.stream[i] = seg_info_host_packed[3 * i];
    tab.start[i] = seg_info_host_packed[3 * i + 1];
    tab.rows[i] = seg_info_host_packed[3 * i + 2];
    tab.first_row[i + 1] = tab.first_row[i] + tab.rows[i];
  }
  if (rows > 0 || lens != nullptr || nzero > 0) {
    TraceScope ts(st, "prep_rows", rows * 8.0, 0.0);
    const int grid = std::max(1, (rows + 255) / 256);
    const cudaError_t e = launch_pdl(prep_rows_kernel, dim3(grid), dim3(256), 0, st, row_stream, row_pos, row_end, tab,
                                     rows, lens, zero, nzero);
    count_launch();
    if (e != cudaSuccess) return DFLASH_E_CUDA;
  }
  return cuda_status(cudaGetLastError());
}

}  // namespace dfl
