// Internal declarations shared by the host and device translation units.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "dflash.h"

namespace dfl {

constexpr int kMaxASeg = 16;   // projections stacked along the output features
constexpr int kMaxBPlane = 8;  // tap planes stacked along the reduction
constexpr int kTileM = 128;    // output features per tile (TMEM lanes)
constexpr int kTileK = 64;     // reduction per pipeline stage (one 128-byte swizzle row)
constexpr int kGemmThreads = 192;
constexpr int kMaxClusterSplit = 8;  // split-K chunks of a tile = one portable cluster

enum EpiKind { EPI_STORE_F32 = 0, EPI_STORE_BF16 = 1, EPI_RESID = 2, EPI_SWIGLU = 3, EPI_HEADS = 4 };
enum HeadKind { HEAD_Q = 0, HEAD_K = 1, HEAD_V = 2 };

// One projection (Q, K or V of one layer) inside a heads epilogue.
struct HeadSeg {
  int kind;                   // HeadKind
  int heads;                  // heads in this projection
  int cap;                    // cache mode: rows per (stream, head); block mode: unused
  int window;                 // cache mode: > 0 -> slot = pos % window (sliding ring)
  const __nv_bfloat16* gain;  // [d] RMSNorm gain (Q and K)
  __nv_bfloat16* dst;         // block mode: [T, heads*d]; cache mode: [S][heads][cap][d]
};

struct EpiArgs {
  void* out;     // STORE_F32 / STORE_BF16 / RESID / SWIGLU: out[t * ldo + m]
  int64_t ldo;
  // heads epilogue
  int head_dim;
  float eps;
  int pos_mode;          // 0: block rows (stream s_begin + t/16, pos lens[s] + t%16); 1: row tables
  int s_begin;
  const int* lens;
  const int* row_stream;
  const int* row_pos;
  const int* row_end;    // rows mode: end position of the row's segment; a sliding-ring
                         // slot is written only by the last W positions of a segment
  const float2* rope;    // [pos][d/2] = (cos, sin)
  HeadSeg seg[kMaxASeg];
  // RESID / STORE_F32: per-tile sums of squares of the written rows,
  // ss_out[m_tile * ss_ld + t] (null: not published), for the RMSNorm that
  // reads the rows next
  float* ss_out;
  int ss_ld;
  // STORE_BF16: per 128-row tile and output column t, the top cand_k of the
  // tile's bf16-rounded outputs (larger value first, ties to the lower row):
  // cand_v / cand_i[(t * m_tiles + m_tile) * cand_k + r]. 0: none.
  int cand_k;
  float* cand_v;
  int* cand_i;
};

struct GemmArgs {
  CUtensorMap a_map[kMaxASeg];    // weights, one map per stacked projection
  CUtensorMap a2_map;             // second weight of a dual (gate/up) GEMM
  CUtensorMap b_map[kMaxBPlane];  // activations, one map per K plane
  int a_seg_tile[kMaxASeg + 1];   // prefix sum of 128-row tiles per projection
  int n_aseg;
  int b_plane_kb;                 // 64-wide reduction blocks per B plane
  int M, N, K;
  int m_tiles, n_tiles, kb_total, ksplit, units;
  int m_tile0;  // the launch covers weight rows [m_tile0 * 128, M); m_tiles of them
  bool no_cluster;
  float* partial;                 // split-K partial tiles, [units][acc][BN][128]
  int* counters;                  // [m_tiles * n_tiles], zero before launch
  int* err;                       // device status word
  EpiArgs epi;
};

// Host-side description of a GEMM D[M, N] = A[M, K] * B[N, K]^T (both
// K-contiguous bf16): A = weights (stacked projections), B = activations
// (optionally K-split over planes).
struct GemmPlan {
  int n_aseg = 0;
  const CUtensorMap* a_maps[kMaxASeg] = {};
  int a_rows[kMaxASeg] = {};
  const CUtensorMap* a2_map = nullptr;  // non-null: dual GEMM
  int n_b = 0;
  const void* b_ptr[kMaxBPlane] = {};
  int64_t ldb = 0;  // elements
  int Kp = 0;       // reduction length of one B plane
  int M = 0, N = 0, K = 0;
  int ksplit = 1;
  int bn = 0;               // token tile width (16, 128 or 256); 0: gemm_bn_for(N)
  int m_tile0 = 0;          // first 128-row tile of the weight this launch covers (M rows from there)
  bool no_cluster = false;  // split-K through global partials even when a cluster would fit
  int epi = EPI_STORE_F32;
  EpiArgs epi_args{};
  const char* name = "gemm";  // trace label
};

// Workspace needed by one GEMM launch (partials and counters), bytes.
size_t gemm_partial_bytes(const GemmPlan& p);
size_t gemm_counter_count(const GemmPlan& p);
int gemm_bn_for(int N);
// The token tile width a plan launches with.
inline int plan_bn(const GemmPlan& p) { return p.bn ? p.bn : gemm_bn_for(p.N); }
// Fixed split of the reduction for a weight matrix (independent of N).
int gemm_choose_ksplit(int m_tiles, int kb_total, int num_sms);
// Encode the TMA map of a K-contiguous bf16 matrix [rows, cols] (row stride ld
// elements) with a box of box_rows x 64 and 128-byte swizzle.
int encode_kmajor_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int64_t ld, int box_rows);
int gemm_launch(const GemmPlan& p, float* partial, int* counters, int* err, int num_sms, cudaStream_t st);

// ---------------------------------------------------------------- small kernels (rows.cu)
// X = embedding rows of [anchor + 15 mask] per stream, with the per-128-
// feature sums of squares of every row, ss[p][T], and (xn != null) the
// rows' RMSNorm with gain g into xn; zero[0, nzero) is cleared (the call's
// split-K counters). A plain launch.
int launch_embed(float* X, float* ss, const __nv_bfloat16* embed, const int* anchors, int S, int H, int V, int mask,
                 int* err, int* zero, int nzero, __nv_bfloat16* xn, const __nv_bfloat16* g, float eps,
                 cudaStream_t st);
// The same sums of squares for rows of a caller-given X [rows, H].
int launch_row_sumsq(float* ss, const float* X, int rows, int H, cudaStream_t st);
int launch_wait_probe(int* err, long long cycles, cudaStream_t st);
// out[r] = bf16(x[src] * rstd * g) with rstd = rsqrt(sum_p ss[p][src] / H +
// eps) from the rows' published per-128-feature sums of squares (parts summed
// in order); src = r, or the r-th mask row (block rows 1..15) when
// mask_rows_only. Elementwise: 8 features a thread.
int launch_rmsnorm_rows(__nv_bfloat16* out, const float* x, const __nv_bfloat16* g, const float* ss, int ss_ld,
                        int rows, int H, float eps, int mask_rows_only, cudaStream_t st);
// Row tables (stream, position) of appended segments (rows > 0), the new
// stream lengths (start + rows of each segment; lens != null) and a cleared
// counter range zero[0, nzero), in one launch. seg_info_host_packed holds
// (stream, start, rows) per segment, on the host.
int launch_prep_rows(int* row_stream, int* row_pos, int* row_end, int* lens, int nseg, int rows,
                     const int* seg_info_host_packed, int* zero, int nzero, cudaStream_t st);
// Segments of a wide K/V-injection pass for kv_rows: segment s covers heads
// [head0[s], head0[s+1]) of the pass and columns [col0[s], ...) of the raw
// projection rows; gain null for V.
struct KvSegs {
  int n;
  int head0[kMaxASeg + 1];
  int64_t col0[kMaxASeg];
  int heads[kMaxASeg];
  int cap[kMaxASeg];
  int window[kMaxASeg];
  const __nv_bfloat16* gain[kMaxASeg];
  __nv_bfloat16* dst[kMaxASeg];
};
// k_norm + RoPE + cache scatter of raw K/V projections y [rows][ld] fp32.
int launch_kv_rows(const float* y, int64_t ld, const KvSegs& segs, const int* row_stream, const int* row_pos,
                   const int* row_end, const float2* rope, int d, float eps, int rows, cudaStream_t st);
// DFlash2's two-tap dynamic convolution on the residual X [16 * S, H] from
// the normed rows h (bf16, [16 * S, H]): z[t] = h[t] . proj^T (2 * groups
// logits, fp32), then X[t] += a0 * h[t - 1] + a1 * h[t] with (a0, a1) the
// softmax of the row's two logits of the channel's group (no row before a
// stream's first).
constexpr int kMaxConvGroups = 32;
int launch_block_conv(float* X, const __nv_bfloat16* h, float* z, const __nv_bfloat16* proj, int S, int H, int groups,
                      cudaStream_t st);
int launch_hidden_norm(__nv_bfloat16* ring, __nv_bfloat16* fused_tmp, const float* y, const float* ss,
                       const __nv_bfloat16* g, const int* row_stream, const int* row_pos, int rows, int H, int R,
                       float eps, cudaStream_t st);

// ---------------------------------------------------------------- attention (attention.cu)
struct AttnArgs {
  const __nv_bfloat16* Q;   // [T, nq*d]
  const __nv_bfloat16* Kb;  // [T, nkv*d]
  const __nv_bfloat16* Vb;  // [T, nkv*d]
  const __nv_bfloat16* Kc;  // [S][nkv][cap][d]
  const __nv_bfloat16* Vc;
  const int* lens;
  int s_begin;
  int cap;
  int window;               // 0: full layer
  int nq, nkv, d;
  int chunk;                // context rows per work unit
  int nchunk;               // chunk slots per (stream, kv head)
  float* part_o;            // [s][nq][nchunk][16][d]
  float* part_ml;           // [s][nq][nchunk][16][2]
  __nv_bfloat16* out;       // [T, nq*d]
  double trace_bytes;       // algorithmic K/V + Q + O bytes (host estimate, for the trace)
  int* err;                 // device status word (bounded waits)
};
int launch_attention(const AttnArgs& a, int s_count, cudaStream_t st);
// Cluster variant for head dimension 128 (attention_cluster.cu): TMA-fed,
// reduce-scatter over distributed shared memory, no partials in global memory.
bool attention_cluster_supported(const AttnArgs& a);
int attention_cluster_maps(CUtensorMap* kmap, CUtensorMap* vmap, const void* kc, const void* vc, int slabs, int cap);
int launch_attention_cluster(const AttnArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap, int s_count,
                             cudaStream_t st);
size_t attn_partial_floats(int s_count, int nq, int nchunk, int d);
// Tensor-memory variant for head dimension 128 and more than four streams a
// call (attention_tc.cu): one CTA per (stream, kv head, key slice) takes the
// kv head's whole query group as one 128-row MMA (tcgen05, S and P*V in
// tensor memory), slices reduced through distributed shared memory.
bool attention_tc_supported(const AttnArgs& a);
int launch_attention_tc(const AttnArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap, int s_count,
                        int num_sms, cudaStream_t st);

// ---------------------------------------------------------------- selection (select.cu)
// Row-wise top-k (k <= 8) from per-tile candidate lists written by a GEMM
// epilogue (EpiArgs::cand_*): rows x tiles lists of k, each sorted.
// Per row of [streams * 15, V] bf16 logits the top-1 softmax probability at
// temperature T (conf), and per stream the leading rows with conf >= min_p.
int launch_draft_stop(const __nv_bfloat16* logits, int streams, int V, float T, float min_p, float* conf, int* len,
                      cudaStream_t st);
int launch_topk_merge(const float* cand_v, const int* cand_i, int rows, int tiles, int k, int* ids, float* vals,
                      cudaStream_t st);
int launch_topk(const __nv_bfloat16* logits, int rows, int V, int k, float T, const float* uniforms, int* ids,
                float* vals, int* sampled, cudaStream_t st);
int launch_verify_greedy(int S, int V, const int* draft, int dld, const __nv_bfloat16* tl, int* accept, int* out,
                         cudaStream_t st);
int launch_verify_sample(int S, int V, const int* draft, int dld, const __nv_bfloat16* tl, const __nv_bfloat16* dl,
                         const float* u, float T, int* accept, int* out, float* stats, cudaStream_t st);

// Launch a kernel with programmatic stream serialization (PDL) on `st`.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// launch bookkeeping
void count_launch(int n = 1);
int cuda_status(cudaError_t e);

// Per-launch timing trace: while enabled, a scope records a CUDA event on
// its stream when it opens and when it closes, with the launch's algorithmic
// bytes and flops.
struct TraceScope {
  TraceScope(cudaStream_t st, const char* name, double bytes, double flops);
  ~TraceScope();
  cudaStream_t st;
  int idx;
};

}  // namespace dfl
