// Row-wise kernels of the hot path: block embedding, RMSNorm of the fp32
// residual into bf16 GEMM operands, the hidden_norm that turns fc's output
// into fused ring rows, and the bookkeeping of appended rows.
//
// Each row is reduced by one CTA in a fixed order (per-thread strided sums,
// then a warp tree, then the warps in order), so results do not depend on
// which other rows share the launch.
#include "internal.h"
#include "ptx.cuh"

namespace dfl {

namespace {

constexpr int kRowThreads = 256;

__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  const int w = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) red[w] = v;
  __syncthreads();
  float t = 0.f;
  const int nw = blockDim.x >> 5;
  for (int i = 0; i < nw; ++i) t += red[i];
  __syncthreads();
  return t;
}

// X[t] = embed[token_t] as fp32; token 16s is the anchor of stream s, the
// other fifteen rows of the block are the mask token [anchor + 15 mask rows].
__global__ void embed_kernel(float* __restrict__ X, const __nv_bfloat16* __restrict__ E, const int* __restrict__ anchors,
                             int H, int V, int mask, int* err) {
  pdl_trigger();
  pdl_wait();
  const int t = blockIdx.x;
  int tok = mask;
  if ((t & 15) == 0) {
    tok = anchors[t >> 4];
    if (tok < 0 || tok >= V) {
      if (threadIdx.x == 0) atomicOr(err, DFLASH_STATUS_BAD_TOKEN);
      tok = 0;
    }
  }
  const __nv_bfloat16* e = E + static_cast<int64_t>(tok) * H;
  float* x = X + static_cast<int64_t>(t) * H;
  for (int i = threadIdx.x; i < H; i += blockDim.x) x[i] = __bfloat162float(e[i]);
}

// out[r] = bf16(x[src] / sqrt(mean(x[src]^2) + eps) * g). The row is held in
// registers (up to kNormVec float4 per thread), all loads issued up front,
// so a row costs one memory round trip. Rows wider than
// kNormVec * 4 * blockDim fall back to a strided second pass.
constexpr int kNormThreads = 512;
constexpr int kNormVec = 4;

__global__ void __launch_bounds__(kNormThreads) rmsnorm_rows_kernel(__nv_bfloat16* __restrict__ out,
                                                                    const float* __restrict__ x,
                                                                    const __nv_bfloat16* __restrict__ g, int H,
                                                                    float eps, int mask_rows_only) {
  __shared__ float red[32];
  pdl_trigger();
  pdl_wait();
  const int r = blockIdx.x;
  const int src = mask_rows_only ? (r / 15) * 16 + 1 + (r % 15) : r;
  const float4* xr = reinterpret_cast<const float4*>(x + static_cast<int64_t>(src) * H);
  const int nv = H >> 2;
  float4 v[kNormVec];
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < kNormVec; ++i) {
    const int j = threadIdx.x + i * kNormThreads;
    v[i] = j < nv ? xr[j] : make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int i = 0; i < kNormVec; ++i) ss += v[i].x * v[i].x + v[i].y * v[i].y + v[i].z * v[i].z + v[i].w * v[i].w;
  for (int j = threadIdx.x + kNormVec * kNormThreads; j < nv; j += kNormThreads) {
    const float4 t = xr[j];
    ss += t.x * t.x + t.y * t.y + t.z * t.z + t.w * t.w;
  }
  const float tot = block_sum(ss, red);
  const float rstd = rsqrtf(tot / static_cast<float>(H) + eps);
  __nv_bfloat162* o = reinterpret_cast<__nv_bfloat162*>(out + static_cast<int64_t>(r) * H);
  const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(g);
#pragma unroll
  for (int i = 0; i < kNormVec; ++i) {
    const int j = threadIdx.x + i * kNormThreads;
    if (j < nv) {
      const float2 ga = __bfloat1622float2(g2[2 * j]);
      const float2 gb = __bfloat1622float2(g2[2 * j + 1]);
      o[2 * j] = __floats2bfloat162_rn(v[i].x * rstd * ga.x, v[i].y * rstd * ga.y);
      o[2 * j + 1] = __floats2bfloat162_rn(v[i].z * rstd * gb.x, v[i].w * rstd * gb.y);
    }
  }
  for (int j = threadIdx.x + kNormVec * kNormThreads; j < nv; j += kNormThreads) {
    const float4 t = xr[j];
    const float2 ga = __bfloat1622float2(g2[2 * j]);
    const float2 gb = __bfloat1622float2(g2[2 * j + 1]);
    o[2 * j] = __floats2bfloat162_rn(t.x * rstd * ga.x, t.y * rstd * ga.y);
    o[2 * j + 1] = __floats2bfloat162_rn(t.z * rstd * gb.x, t.w * rstd * gb.y);
  }
}

// fused = bf16(RMSNorm(y) * hidden_norm): written to the ring slot of the
// row's (stream, position) and to a dense staging copy for K/V injection.
__global__ void hidden_norm_kernel(__nv_bfloat16* __restrict__ ring, __nv_bfloat16* __restrict__ fused_tmp,
                                   const float* __restrict__ y, const __nv_bfloat16* __restrict__ g,
                                   const int* __restrict__ row_stream, const int* __restrict__ row_pos, int H, int R,
                                   float eps) {
  __shared__ float red[32];
  pdl_trigger();
  pdl_wait();
  const int r = blockIdx.x;
  const float* yr = y + static_cast<int64_t>(r) * H;
  float ss = 0.f;
  for (int i = threadIdx.x; i < H; i += blockDim.x) {
    const float v = yr[i];
    ss += v * v;
  }
  const float tot = block_sum(ss, red);
  const float rstd = rsqrtf(tot / static_cast<float>(H) + eps);
  __nv_bfloat16* dr = ring + (static_cast<int64_t>(row_stream[r]) * R + row_pos[r]) * H;
  __nv_bfloat16* dt = fused_tmp + static_cast<int64_t>(r) * H;
  for (int i = threadIdx.x; i < H; i += blockDim.x) {
    const __nv_bfloat16 b = __float2bfloat16_rn(yr[i] * rstd * __bfloat162float(g[i]));
    dr[i] = b;
    dt[i] = b;
  }
}

struct SegTable {
  int n;
  int stream[256];
  int start[256];
  int rows[256];
  int first_row[257];
};

__global__ void prep_rows_kernel(int* __restrict__ row_stream, int* __restrict__ row_pos, int* __restrict__ row_end,
                                 const SegTable tab, int total) {
  pdl_trigger();
  pdl_wait();
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= total) return;
  int s = 0;
  while (s + 1 < tab.n && r >= tab.first_row[s + 1]) ++s;
  row_stream[r] = tab.stream[s];
  row_pos[r] = tab.start[s] + (r - tab.first_row[s]);
  row_end[r] = tab.start[s] + tab.rows[s];
}

__global__ void set_lens_kernel(int* __restrict__ lens, const SegTable tab) {
  pdl_trigger();
  pdl_wait();
  const int i = threadIdx.x;
  if (i < tab.n) lens[tab.stream[i]] = tab.start[i] + tab.rows[i];
}

}  // namespace

int launch_embed(float* X, const __nv_bfloat16* embed, const int* anchors, int S, int H, int V, int mask, int* err,
                 cudaStream_t st) {
  TraceScope ts(st, "embed", static_cast<double>(S) * 16 * H * 6, 0.0);
  const cudaError_t e = launch_pdl(embed_kernel, dim3(S * 16), dim3(kRowThreads), 0, st, X, embed, anchors, H, V, mask, err);
  count_launch();
  return cuda_status(e);
}

int launch_rmsnorm_rows(__nv_bfloat16* out, const float* x, const __nv_bfloat16* g, int rows, int H, float eps,
                        int mask_rows_only, cudaStream_t st) {
  TraceScope ts(st, "rmsnorm", static_cast<double>(rows) * H * 6, 0.0);
  const cudaError_t e =
      launch_pdl(rmsnorm_rows_kernel, dim3(rows), dim3(kNormThreads), 0, st, out, x, g, H, eps, mask_rows_only);
  count_launch();
  return cuda_status(e);
}

int launch_hidden_norm(__nv_bfloat16* ring, __nv_bfloat16* fused_tmp, const float* y, const __nv_bfloat16* g,
                       const int* row_stream, const int* row_pos, int rows, int H, int R, float eps, cudaStream_t st) {
  TraceScope ts(st, "hidden_norm", static_cast<double>(rows) * H * 8, 0.0);
  const cudaError_t e = launch_pdl(hidden_norm_kernel, dim3(rows), dim3(kRowThreads), 0, st, ring, fused_tmp, y, g,
                                   row_stream, row_pos, H, R, eps);
  count_launch();
  return cuda_status(e);
}

// seg_info_host_packed: 3*nseg ints (stream, start, rows) on the host.
int launch_prep_rows(int* row_stream, int* row_pos, int* row_end, int* lens, int nseg, int rows,
                     const int* seg_info_host_packed, cudaStream_t st) {
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
  if (rows > 0) {
    TraceScope ts(st, "prep_rows", rows * 8.0, 0.0);
    const cudaError_t e =
        launch_pdl(prep_rows_kernel, dim3((rows + 255) / 256), dim3(256), 0, st, row_stream, row_pos, row_end, tab, rows);
    count_launch();
    if (e != cudaSuccess) return DFLASH_E_CUDA;
  }
  if (lens) {
    TraceScope ts(st, "set_lens", nseg * 4.0, 0.0);
    const cudaError_t e = launch_pdl(set_lens_kernel, dim3(1), dim3(256), 0, st, lens, tab);
    count_launch();
    if (e != cudaSuccess) return DFLASH_E_CUDA;
  }
  return cuda_status(cudaGetLastError());
}

}  // namespace dfl
