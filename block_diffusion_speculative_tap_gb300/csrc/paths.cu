// DFlash2 candidate-path selector: the one consistent path through the
// per-position top-k candidates of a drafted block.
//
// "DFlash 解碼加速" explainer, section 五 ("Candidate path selector"):
// DFlash 2 keeps the top-k candidates at every position, a light selector
// scores adjacent candidate pairs, and one consistent path is chosen
// (selector_top_k 16, selector_rank 256 in the public DFlash2 config).
// TensorFold #1851, item 1: with no codebooks (rank 0) the edge term is zero.
// Reading: path score = the candidates' node scores (the drafter's logits)
// plus, for every adjacent pair, the rank-r bilinear form <U[id_i], W[id_i+1]>
// of per-token codebooks U, W [V, r]; the best path by the max-sum recursion
// (Viterbi), ties to the lower candidate index.
//
// Two kernels:
//   selector_edges_kernel: one CTA per (stream, adjacent pair of positions);
//     the two positions' codebook rows go to shared memory (padded rows, so
//     the 16 rows a warp reads at one column sit in 16 banks) and each thread
//     forms one pair's dot product in fp32, ascending over the rank.
//   selector_path_kernel: one warp per stream; lane b holds the best score
//     of a path ending in candidate b, the recursion takes each step's
//     maximum over the previous position's lanes by shuffles, and lane 0
//     walks the back-pointers.
//
// Tree drafting and tree verification (TensorFold #1851: per-stream trees;
// with no codebooks the trees come from each depth's marginals; the
// explainer's section 四: the greedy rule). Reading: the root is the anchor,
// every node of depth j - 1 has the top-b_j candidates of mask row j as
// children in candidate order, nodes numbered breadth first. Then a node of
// depth j with index l inside its depth has candidate index l % b_j and
// parent l / b_j inside depth j - 1 (mixed radix), so the tree is built with
// no search:
//   tree_build_kernel: one thread a node: token, parent, depth and the row of
//     the ancestor-or-self mask a target applies to score the tree in one
//     pass.
//   tree verification: the vocabulary arg-max scan over every node's target
//     row (the same scan as greedy verification), then tree_walk_kernel: one
//     warp a stream, lane c tests the current node's child c against the
//     arg-max, the lowest matching lane is followed.
#include <float.h>

#include "internal.h"
#include "ptx.cuh"

namespace dfl {

namespace {

constexpr int kSelEdgeThreads = 256;  // >= DFLASH_MAX_TOPK^2 pairs

__global__ void __launch_bounds__(kSelEdgeThreads)
    selector_edges_kernel(const int* __restrict__ cand_ids, int P, int k, int V, int r,
                          const __nv_bfloat16* __restrict__ U, const __nv_bfloat16* __restrict__ W,
                          float* __restrict__ E) {
  extern __shared__ uint32_t rows[];  // [2k][r/2 + 1] bf16 pairs: U rows of position i, then W rows of i+1
  pdl_trigger();
  pdl_wait();
  const int s = blockIdx.x, i = blockIdx.y;  // streams on x: no 65535 limit
  const int words = r / 2, stride = words + 1;
  const int* ids_i = cand_ids + (static_cast<int64_t>(s) * P + i) * k;
  // stage: row q < k is U[c(i, q)], row k + q is W[c(i+1, q)]; an id outside
  // [0, V) is not a candidate and its row counts as zero
  const int vec = r / 8;  // 16-byte pieces a row
  for (int t = threadIdx.x; t < 2 * k * vec; t += blockDim.x) {
    const int row = t / vec, piece = t - row * vec;
    const int q = row < k ? row : row - k;
    const int id = ids_i[(row < k ? 0 : k) + q];
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (id >= 0 && id < V) {
      const __nv_bfloat16* src = (row < k ? U : W) + static_cast<int64_t>(id) * r + piece * 8;
      v = *reinterpret_cast<const uint4*>(src);
    }
    uint32_t* dst = rows + row * stride + piece * 4;
    dst[0] = v.x;
    dst[1] = v.y;
    dst[2] = v.z;
    dst[3] = v.w;
  }
  __syncthreads();
  const int a = threadIdx.x / k, b = threadIdx.x - (threadIdx.x / k) * k;
  if (a >= k) return;
  const uint32_t* ua = rows + a * stride;
  const uint32_t* wb = rows + (k + b) * stride;
  float acc = 0.f;
  for (int j = 0; j < words; ++j) {
    const uint32_t x = ua[j], y = wb[j];
    const float2 fx = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&x));
    const float2 fy = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&y));
    acc = fmaf(fx.x, fy.x, acc);
    acc = fmaf(fx.y, fy.y, acc);
  }
  E[((static_cast<int64_t>(s) * (P - 1) + i) * k + a) * k + b] = acc;
}

__global__ void __launch_bounds__(32)
    selector_path_kernel(const int* __restrict__ cand_ids, const float* __restrict__ cand_vals, int P, int k, int V,
                         const float* __restrict__ E, int* __restrict__ path_ids, int* __restrict__ path_ranks,
                         float* __restrict__ path_score) {
  __shared__ unsigned char back[DFLASH_BLOCK][DFLASH_MAX_TOPK];
  pdl_trigger();
  pdl_wait();
  const int s = blockIdx.x, b = threadIdx.x;
  const int* ids = cand_ids + static_cast<int64_t>(s) * P * k;
  const float* vals = cand_vals + static_cast<int64_t>(s) * P * k;
  auto node = [&](int i) -> float {
    if (b >= k) return -INFINITY;
    const int id = ids[i * k + b];
    return (id >= 0 && id < V) ? vals[i * k + b] : -INFINITY;
  };
  float F = node(0);
  for (int i = 1; i < P; ++i) {
    const float* Ei = E + (static_cast<int64_t>(s) * (P - 1) + (i - 1)) * k * k;
    float best = -INFINITY;
    int arg = 0;
    for (int a = 0; a < k; ++a) {
      const float fa = __shfl_sync(0xffffffffu, F, a);
      const float v = b < k ? fa + Ei[a * k + b] : -INFINITY;
      if (v > best) {  // the lower index keeps a tie
        best = v;
        arg = a;
      }
    }
    F = node(i) + best;
    if (b < k) back[i][b] = static_cast<unsigned char>(arg);
  }
  // the best last candidate, ties to the lower index
  float m = F;
  int arg = b < k ? b : k;
  for (int off = 16; off >= 1; off >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
    const int a2 = __shfl_xor_sync(0xffffffffu, arg, off);
    if (m2 > m || (m2 == m && a2 < arg)) {
      m = m2;
      arg = a2;
    }
  }
  __syncwarp();
  if (b != 0) return;
  int* out_ids = path_ids + static_cast<int64_t>(s) * P;
  int* out_ranks = path_ranks ? path_ranks + static_cast<int64_t>(s) * P : nullptr;
  if (m == -INFINITY) {  // some position has no valid candidate
    for (int i = 0; i < P; ++i) {
      out_ids[i] = -1;
      if (out_ranks) out_ranks[i] = -1;
    }
    if (path_score) path_score[s] = -INFINITY;
    return;
  }
  int cur = arg;
  for (int i = P - 1; i >= 0; --i) {
    out_ids[i] = ids[i * k + cur];
    if (out_ranks) out_ranks[i] = cur;
    if (i > 0) cur = back[i][cur];
  }
  if (path_score) path_score[s] = m;
}

struct TreeShape {
  int depth;                         // D: depths 1..D below the root
  int n;                             // nodes, the root included
  int width[DFLASH_BLOCK];           // width[j] = b_j, j = 1..D
  int offset[DFLASH_BLOCK + 1];      // first node of depth j; offset[D + 1] = n
};

__device__ __forceinline__ int tree_depth_of(const TreeShape& t, int n) {
  int j = 0;
  while (j < t.depth && n >= t.offset[j + 1]) ++j;
  return j;
}

__global__ void __launch_bounds__(256)
    tree_build_kernel(TreeShape t, int k, const int* __restrict__ anchors, const int* __restrict__ topk_ids,
                      int* __restrict__ tokens, int* __restrict__ parents, int* __restrict__ depths,
                      uint32_t* __restrict__ mask, int mask_words) {
  pdl_trigger();
  pdl_wait();
  const int s = blockIdx.x;
  for (int n = threadIdx.x; n < t.n; n += blockDim.x) {
    const int j = tree_depth_of(t, n);
    int token, parent;
    if (j == 0) {
      token = anchors[s];
      parent = -1;
    } else {
      const int l = n - t.offset[j];
      token = topk_ids[(static_cast<int64_t>(s) * (DFLASH_BLOCK - 1) + (j - 1)) * k + l % t.width[j]];
      parent = t.offset[j - 1] + l / t.width[j];
    }
    const int64_t o = static_cast<int64_t>(s) * t.n + n;
    tokens[o] = token;
    if (parents) parents[o] = parent;
    if (depths) depths[o] = j;
    if (mask) {
      // ancestors: at depth i < j the index inside depth i is l / (b_{i+1} ... b_j)
      int anc[DFLASH_BLOCK];
      int l = n - t.offset[j];
      for (int i = j; i >= 0; --i) {
        anc[i] = t.offset[i] + l;
        if (i > 0) l /= t.width[i];
      }
      uint32_t* row = mask + o * mask_words;
      for (int w = 0; w < mask_words; ++w) {
        uint32_t bits = 0u;
        for (int i = 0; i <= j; ++i)
          if ((anc[i] >> 5) == w) bits |= 1u << (anc[i] & 31);
        row[w] = bits;
      }
    }
  }
}

__global__ void __launch_bounds__(32)
    tree_walk_kernel(TreeShape t, const int* __restrict__ tokens, const int* __restrict__ amax,
                     int* __restrict__ accept, int* __restrict__ out, int* __restrict__ node_out) {
  pdl_trigger();
  pdl_wait();
  const int s = blockIdx.x, lane = threadIdx.x;
  const int* tk = tokens + static_cast<int64_t>(s) * t.n;
  const int* am = amax + static_cast<int64_t>(s) * t.n;
  int cur = 0, j = 0, mine = -1;  // lane i keeps the token accepted at depth i + 1
  while (j < t.depth) {
    const int target = am[cur];
    const int b = t.width[j + 1];
    const int first = t.offset[j + 1] + (cur - t.offset[j]) * b;
    const bool hit = lane < b && tk[first + lane] == target;
    const unsigned m = __ballot_sync(0xffffffffu, hit);
    if (!m) break;
    cur = first + __ffs(m) - 1;
    if (lane == j) mine = target;
    ++j;
  }
  const int bonus = am[cur];
  if (lane < DFLASH_BLOCK) out[static_cast<int64_t>(s) * DFLASH_BLOCK + lane] = lane < j ? mine : (lane == j ? bonus : -1);
  if (lane == 0) {
    accept[s] = j;
    if (node_out) node_out[s] = cur;
  }
}

// Shape of a tree of the given depth and widths; DFLASH_E_INVALID_ARG when a
// width is outside [1, k], the depth outside [1, 15], or the tree has more
// than DFLASH_MAX_TREE_NODES nodes.
int tree_shape(int depth, const int32_t* widths, int k, TreeShape* t) {
  if (depth < 1 || depth > DFLASH_BLOCK - 1 || !widths || k < 1 || k > DFLASH_MAX_TOPK) return DFLASH_E_INVALID_ARG;
  *t = TreeShape{};
  t->depth = depth;
  t->offset[0] = 0;
  t->offset[1] = 1;
  int64_t level = 1, n = 1;
  for (int j = 1; j <= depth; ++j) {
    const int b = widths[j - 1];
    if (b < 1 || b > k) return DFLASH_E_INVALID_ARG;
    t->width[j] = b;
    level *= b;
    n += level;
    if (n > DFLASH_MAX_TREE_NODES) return DFLASH_E_INVALID_ARG;
    t->offset[j + 1] = static_cast<int>(n);
  }
  t->n = static_cast<int>(n);
  return DFLASH_OK;
}

}  // namespace

size_t selector_ws_bytes(int streams, int positions, int k) {
  if (streams <= 0 || positions <= 1) return 0;
  return static_cast<size_t>(streams) * (positions - 1) * k * k * sizeof(float);
}

int launch_select_path(int S, int P, int k, int V, int r, const int* cand_ids, const float* cand_vals,
                       const __nv_bfloat16* U, const __nv_bfloat16* W, int* path_ids, int* path_ranks,
                       float* path_score, float* E, cudaStream_t st) {
  if (S <= 0) return DFLASH_OK;
  if (P > 1) {
    const size_t smem = static_cast<size_t>(2 * k) * (r / 2 + 1) * sizeof(uint32_t);
    const double bytes = static_cast<double>(S) * (P - 1) * (2.0 * k * r * 2 + k * 4 * 2 + k * k * 4.0);
    TraceScope ts(st, "selector.edges", bytes, 2.0 * S * (P - 1) * k * k * r);
    const cudaError_t e = launch_pdl(selector_edges_kernel, dim3(S, P - 1), dim3(kSelEdgeThreads), smem, st,
                                     cand_ids, P, k, V, r, U, W, E);
    count_launch();
    if (e != cudaSuccess) return DFLASH_E_CUDA;
  }
  {
    const double bytes = static_cast<double>(S) * (P * k * 8.0 + (P - 1) * k * k * 4.0 + P * 8.0 + 4.0);
    TraceScope ts(st, "selector.path", bytes, 0.0);
    const cudaError_t e = launch_pdl(selector_path_kernel, dim3(S), dim3(32), 0, st, cand_ids, cand_vals, P, k, V,
                                     static_cast<const float*>(E), path_ids, path_ranks, path_score);
    count_launch();
    if (e != cudaSuccess) return DFLASH_E_CUDA;
  }
  return DFLASH_OK;
}

}  // namespace dfl

extern "C" int dflash_select_path_workspace_bytes(int streams, int positions, int k, size_t* bytes) {
  if (!bytes || streams < 0 || positions < 1 || positions > DFLASH_BLOCK || k < 1 || k > DFLASH_MAX_TOPK)
    return DFLASH_E_INVALID_ARG;
  *bytes = dfl::selector_ws_bytes(streams, positions, k);
  return DFLASH_OK;
}

extern "C" int dflash_select_path(int streams, int positions, int k, int vocab, int rank, const int32_t* cand_ids,
                                  const float* cand_vals, const void* U, const void* W, int32_t* path_ids,
                                  int32_t* path_ranks, float* path_score, void* ws, size_t ws_bytes,
                                  dflash_stream_t stream) {
  if (streams < 0 || positions < 1 || positions > DFLASH_BLOCK || k < 1 || k > DFLASH_MAX_TOPK || vocab < 1 ||
      rank < 0 || rank > DFLASH_MAX_SELECTOR_RANK || rank % 8)
    return DFLASH_E_INVALID_ARG;
  if (streams == 0) return DFLASH_OK;
  if (!cand_ids || !cand_vals || !path_ids) return DFLASH_E_INVALID_ARG;
  if (positions > 1 && rank > 0) {
    if (!U || !W || (reinterpret_cast<uintptr_t>(U) & 15u) || (reinterpret_cast<uintptr_t>(W) & 15u))
      return DFLASH_E_INVALID_ARG;
  }
  const size_t need = dfl::selector_ws_bytes(streams, positions, k);
  if (need && (!ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 15u))) return DFLASH_E_WORKSPACE;
  return dfl::launch_select_path(streams, positions, k, vocab, rank, cand_ids, cand_vals,
                                 static_cast<const __nv_bfloat16*>(U), static_cast<const __nv_bfloat16*>(W), path_ids,
                                 path_ranks, path_score, static_cast<float*>(ws),
                                 reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int dflash_tree_size(int depth, const int32_t* widths, int k, int* nodes) {
  if (!nodes) return DFLASH_E_INVALID_ARG;
  dfl::TreeShape t;
  const int rc = dfl::tree_shape(depth, widths, k, &t);
  if (rc) return rc;
  *nodes = t.n;
  return DFLASH_OK;
}

extern "C" int dflash_tree_build(int streams, int depth, const int32_t* widths, int k, const int32_t* anchors,
                                 const int32_t* topk_ids, int32_t* node_tokens, int32_t* node_parent,
                                 int32_t* node_depth, uint32_t* node_mask, dflash_stream_t stream) {
  if (streams < 0) return DFLASH_E_INVALID_ARG;
  dfl::TreeShape t;
  const int rc = dfl::tree_shape(depth, widths, k, &t);
  if (rc) return rc;
  if (streams == 0) return DFLASH_OK;
  if (!anchors || !topk_ids || !node_tokens) return DFLASH_E_INVALID_ARG;
  const int words = (t.n + 31) / 32;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const double bytes = static_cast<double>(streams) *
                       (4.0 + depth * k * 4.0 + t.n * 4.0 * (1 + (node_parent != nullptr) + (node_depth != nullptr)) +
                        (node_mask ? t.n * words * 4.0 : 0.0));
  dfl::TraceScope ts(st, "tree.build", bytes, 0.0);
  const cudaError_t e = dfl::launch_pdl(dfl::tree_build_kernel, dim3(streams), dim3(256), 0, st, t, k, anchors,
                                        topk_ids, node_tokens, node_parent, node_depth, node_mask, words);
  dfl::count_launch();
  return e == cudaSuccess ? DFLASH_OK : DFLASH_E_CUDA;
}

extern "C" int dflash_tree_verify_workspace_bytes(int streams, int nodes, size_t* bytes) {
  if (!bytes || streams < 0 || nodes < 1 || nodes > DFLASH_MAX_TREE_NODES) return DFLASH_E_INVALID_ARG;
  *bytes = static_cast<size_t>(streams) * nodes * (sizeof(int) + sizeof(float));
  return DFLASH_OK;
}

extern "C" int dflash_tree_verify(int streams, int depth, const int32_t* widths, int vocab, const int32_t* node_tokens,
                                  const void* target_logits, int32_t* accept_len, int32_t* out_tokens,
                                  int32_t* accept_node, void* ws, size_t ws_bytes, dflash_stream_t stream) {
  if (streams < 0 || vocab < 8 || vocab % 8) return DFLASH_E_INVALID_ARG;
  dfl::TreeShape t;
  const int rc = dfl::tree_shape(depth, widths, DFLASH_MAX_TOPK, &t);
  if (rc) return rc;
  if (streams == 0) return DFLASH_OK;
  if (!node_tokens || !target_logits || !accept_len || !out_tokens || (reinterpret_cast<uintptr_t>(target_logits) & 15u))
    return DFLASH_E_INVALID_ARG;
  const size_t need = static_cast<size_t>(streams) * t.n * (sizeof(int) + sizeof(float));
  if (!ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 15u)) return DFLASH_E_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int* amax = static_cast<int*>(ws);
  float* vals = reinterpret_cast<float*>(amax + static_cast<size_t>(streams) * t.n);
  int r = dfl::launch_topk(static_cast<const __nv_bfloat16*>(target_logits), streams * t.n, vocab, 1, 1.0f, nullptr,
                           amax, vals, nullptr, st);
  if (r) return r;
  dfl::TraceScope ts(st, "tree.walk", static_cast<double>(streams) * (t.n * 8.0 + DFLASH_BLOCK * 4.0 + 8.0), 0.0);
  const cudaError_t e = dfl::launch_pdl(dfl::tree_walk_kernel, dim3(streams), dim3(32), 0, st, t, node_tokens,
                                        static_cast<const int*>(amax), accept_len, out_tokens, accept_node);
  dfl::count_launch();
  return e == cudaSuccess ? DFLASH_OK : DFLASH_E_CUDA;
}
