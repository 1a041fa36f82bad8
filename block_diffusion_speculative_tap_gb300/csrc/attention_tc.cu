// Block attention on the fifth-generation tensor cores (tcgen05, scores and
// outputs in tensor memory) for head dimension 128 when a draft call carries
// more than four streams.
//
// One CTA per (stream, kv head, key slice) takes all G query heads of the kv
// head at once: their 16 block rows each make the 16*G <= 128 rows of the
// MMA's M side (rows past 16*G are zero), so every K/V tile is read once for
// the whole group. The visible context keys are split evenly over the CS CTAs
// of a thread-block cluster; the last CTA also takes the block's own 16 keys.
//
// A 128-row MMA of 16 k-steps takes about 120 cycles on GB300 whether it is
// 16, 64 or 128 columns wide (measured), so the scores of two 64-key tiles
// are taken in one 128-column MMA: a step is 128 keys. K and V stream through four rings of 64-key slots (K
// dims 0-63, K dims 64-127, V dims 0-63, V dims 64-127) so that a step's two
// tiles sit in adjacent slots and read as one 128-row operand. Both A operands
// live in tensor memory (row i of A in lane i, two bf16 of consecutive k in
// each 32-bit column): the softmax warps copy Q there once and write P there.
//
// Roles (608 threads):
//   warp 0     TMA producer: 64-key tiles of K and V (head-major cache, 3-D
//              tensor maps, 128-byte swizzle) into the rings, and the block's
//              K/V.
//   warp 1     tensor-memory owner and score MMA issuer: S = Q K^T of step
//              u+1 as soon as the softmax warps have read step u's scores.
//   warp 2     output MMA issuer: O += P_u V_u (V read MN-major) once the
//              softmax warps have written P_u. Issuing blocks while the
//              tensor pipe is busy, so the two kinds of MMA have a thread
//              each: the next scores never queue behind the previous P*V.
//   warps 3-18 softmax: four warps a tensor-memory lane quadrant, each taking
//              32 of a step's keys for the quadrant's 32 rows (thread r of a
//              warp owns row r). The four share their step maximum through
//              shared memory and a named barrier; each keeps its keys' sum and
//              the maximum the probabilities are taken against (log2 domain),
//              and writes its keys of P as bf16 into one of two P buffers in
//              tensor memory. The output accumulates over the steps in tensor
//              memory; the maximum in use moves (and the row's output and sum
//              are rescaled in place, each warp its 32 output columns) only
//              when a step's maximum exceeds it by more than kRescaleLog2, so
//              a probability never exceeds 2^kRescaleLog2. Warps whose rows
//              are all padding take no part.
// The CTAs of a cluster then reduce-scatter their (max, sum, output) rows
// through distributed shared memory in rank order and write bf16 rows.
// P enters P*V as bf16; the sum uses fp32 P. Every wait is bounded.
#include <mutex>
#include <utility>
#include <vector>

#include "internal.h"
#include "ptx.cuh"

namespace dfl {

namespace {

constexpr int kD = 128;
constexpr int kTK = 64;                  // keys a context tile (one TMA box, one ring slot)
constexpr int kSK = 2 * kTK;             // keys a step: two tiles, one 128-column score MMA
constexpr int kBK = 16;                  // the block's own keys
constexpr int kStages = 6;               // ring slots (even: a step's tiles take adjacent slots)
constexpr int kRows = 128;               // MMA rows: 16 query rows x G, zero-padded
constexpr int kSlot = kTK * 128;         // 64 keys x 64 dims bf16 (8 KiB)
constexpr int kRing = kStages * kSlot;   // one ring (48 KiB)
constexpr int kTileBytes = 4 * kSlot;    // a tile's K and V (32 KiB)
constexpr int kBSub = kBK * 128;         // 16 keys x 64 dims (2 KiB)
constexpr int kPartLd = kD + 4;          // fp32 partial row stride
constexpr int kParts = 4;                // softmax warps a lane quadrant
constexpr int kThreads = 96 + 128 * kParts;
// tensor-memory columns: the step's scores (0..127), the output (128..255),
// Q as the score MMAs' A operand (64 columns: 128 dims as bf16 pairs) and two
// P buffers (64 columns each: 128 keys as bf16 pairs)
constexpr int kColS = 0;
constexpr int kColO = 128;
constexpr int kColQ = 256;
constexpr int kColP = 320;
// All of an SM's tensor memory: the CTA's 207 KB of shared memory leave no
// room on its SM for a CTA of the other tensor-memory user (every GEMM CTA
// takes at least 93 KB), so the allocation never waits on another kernel.
constexpr int kTmemCols = 512;
constexpr float kRescaleLog2 = 8.f;      // a row's maximum in use moves only past this margin

struct TcSmem {
  static constexpr int kKlo = 0;
  static constexpr int kKhi = kKlo + kRing;
  static constexpr int kVlo = kKhi + kRing;
  static constexpr int kVhi = kVlo + kRing;
  static constexpr int kBlock = kVhi + kRing;  // the block's K lo, K hi, V lo, V hi
  static constexpr int kBar = kBlock + 4 * kBSub;
  static constexpr int kXchg = kBar + 256;                        // [4 quadrants][kParts][2][32] step maxima
  static constexpr int kLPart = kXchg + 4 * kParts * 2 * 32 * 4;  // [kParts][128] row sums
  static constexpr int kBytes = kLPart + kParts * kRows * 4;
};
static_assert(kStages % 2 == 0, "a step's two tiles must sit in adjacent ring slots");
static_assert(TcSmem::kKhi % 1024 == 0 && TcSmem::kBlock % 1024 == 0,
              "swizzled tiles must start on 1024-byte boundaries");
static_assert(sizeof(float) * (kRows * kPartLd + kRows * 2) <= 4 * kRing,
              "the partials must fit the ring memory");
static_assert(8 * (2 * kStages + 11) <= 256, "the barriers must fit their region");
constexpr int kSmemLaunch = TcSmem::kBytes + 1024;

// MN-major operand stored with the 128-byte swizzle, as TMA writes a tile of
// rows that each hold 64 consecutive MN elements: 8 rows (8 consecutive K)
// make a 1024-byte atom; `lbo` bytes separate 64-element blocks along MN and
// 1024 bytes separate 8-row groups along K. Fields as in sdesc_sw128.
__device__ __forceinline__ uint64_t sdesc_sw128_mn(uint32_t saddr, uint32_t lbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>(1024u >> 4) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(2u) << 61;
  return d;
}

// kind::f16 instruction descriptor bit 16: B is MN-major.
constexpr uint32_t kIdescBTransposed = 1u << 16;

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

// Load 32 consecutive 32-bit tensor-memory columns of this warp's 32 lanes
// (one lane per thread); the caller waits with tmem_wait_ld before use.
__device__ __forceinline__ void tmem_ld32_async(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 2^x by the SFU's approximate base-2 exponential (relative error a few
// units of fp32's last place; -inf gives +0). P is rounded to bf16 after it.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Store 16 consecutive 32-bit tensor-memory columns of this warp's 32 lanes
// and wait until the stores are done.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
      "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])),
      "r"(__float_as_uint(v[11])), "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])),
      "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15]))
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Store 16 consecutive 32-bit tensor-memory columns of this warp's 32 lanes
// (one lane per thread); the caller waits with tmem_wait_st.
__device__ __forceinline__ void tmem_st16u(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// D[tmem] (+)= A[tmem] * B[smem], issued by one thread: A's row i is lane i
// of the columns from a_tmem on, two bf16 of consecutive k a column.
__device__ __forceinline__ void umma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

struct TcArgs {
  CUtensorMap kmap;   // cache K: 3-D [S*nkv][cap][128], box {64, 64, 1}
  CUtensorMap vmap;
  CUtensorMap kbmap;  // block K: 2-D [T][nkv*128], box {64, 16}
  CUtensorMap vbmap;
  AttnArgs a;
};

template <int CS>
__global__ void __launch_bounds__(kThreads, 1) attn_tc_kernel(const __grid_constant__ TcArgs P) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const AttnArgs& a = P.a;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + TcSmem::kBar);
  uint64_t* full = bars;                  // [kStages] a context tile landed in its ring slot
  uint64_t* empty = bars + kStages;       // [kStages] the MMAs reading the slot are done
  uint64_t* s_full = bars + 2 * kStages;  // the step's scores are in tensor memory
  uint64_t* s_empty = s_full + 1;         // the softmax warps have read them
  uint64_t* p_full = s_full + 2;          // [2] P written to tensor memory (and the output rescaled)
  uint64_t* o_full = s_full + 4;          // [2] P*V of a step using P buffer b has landed in the output
  uint64_t* blk_full = s_full + 6;        // the block's K/V landed
  uint64_t* q_tm = s_full + 7;            // the Q rows are in tensor memory
  uint64_t* drain = s_full + 8;           // [2] every MMA of either issuer is done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(s_full + 10);
  int* abort_word = reinterpret_cast<int*>(tmem_slot + 1);
  const uint32_t sbase = smem_u32(smem);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = crank();
  const int kvh = blockIdx.y, si = blockIdx.z;
  const int G = a.nq / a.nkv;
  const int rows = 16 * G;
  const int nact = (rows + 31) / 32;  // lane quadrants with real rows: 0 .. nact-1 (kParts softmax warps each)
  int* err = a.err;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_empty, 128 * nact);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&p_full[b], 128 * nact);
      mbar_init(&o_full[b], 1);
    }
    mbar_init(blk_full, 1);
    mbar_init(q_tm, 128 * nact);
    mbar_init(&drain[0], 1);
    mbar_init(&drain[1], 1);
    *abort_word = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_trigger();
  // The context K/V tiles and the stream lengths come from earlier fills,
  // complete before a draft call's first kernel starts (that kernel is
  // launched without programmatic dependence): the producer loads the first
  // slots before the PDL wait. Q and the block's own K/V come from the
  // Q/K/V GEMM, after it.
  const bool producer = warp == 0 && lane == 0;
  if (!producer) pdl_wait();

  const int s = a.s_begin + si;
  const int C = a.lens[s];
  const int nvis = a.window > 0 ? min(C, a.window) : C;
  const int k0 = static_cast<int>(static_cast<long long>(nvis) * rank / CS);
  const int k1 = static_cast<int>(static_cast<long long>(nvis) * (rank + 1) / CS);
  const int nkeys = k1 - k0;
  const int nctx = (nkeys + kTK - 1) / kTK;  // context tiles
  const int nsc = (nctx + 1) / 2;            // context steps: tiles 2j and 2j+1
  const bool has_block = rank == CS - 1;
  const int nS = nsc + (has_block ? 1 : 0);  // step nsc is the block's own keys
  const int slab = s * a.nkv + kvh;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      auto load_tile = [&](int t) {
        const int sl = t % kStages;
        const int row = k0 + t * kTK;
        mbar_arrive_expect_tx(&full[sl], kTileBytes);
        tma3d(sbase + TcSmem::kKlo + sl * kSlot, &P.kmap, &full[sl], 0, row, slab);
        tma3d(sbase + TcSmem::kKhi + sl * kSlot, &P.kmap, &full[sl], 64, row, slab);
        tma3d(sbase + TcSmem::kVlo + sl * kSlot, &P.vmap, &full[sl], 0, row, slab);
        tma3d(sbase + TcSmem::kVhi + sl * kSlot, &P.vmap, &full[sl], 64, row, slab);
      };
      const int npre = nctx < kStages ? nctx : kStages;
      for (int t = 0; t < npre; ++t) load_tile(t);
      pdl_wait();
      if (has_block) {
        mbar_arrive_expect_tx(blk_full, 4 * kBSub);
        const uint32_t b = sbase + TcSmem::kBlock;
        tma2d(b, &P.kbmap, blk_full, kvh * kD, 16 * si);
        tma2d(b + kBSub, &P.kbmap, blk_full, kvh * kD + 64, 16 * si);
        tma2d(b + 2 * kBSub, &P.vbmap, blk_full, kvh * kD, 16 * si);
        tma2d(b + 3 * kBSub, &P.vbmap, blk_full, kvh * kD + 64, 16 * si);
      }
      for (int t = npre; t < nctx; ++t) {
        const int sl = t % kStages;
        if (!mbar_wait(&empty[sl], ((t / kStages) & 1) ^ 1u, err, DFLASH_STATUS_TIMEOUT, abort_word)) break;
        load_tile(t);
      }
      // no copy may still be landing when the ring memory is reused below
      for (int sl = 0; sl < kStages && sl < nctx; ++sl) {
        const int last = sl + ((nctx - 1 - sl) / kStages) * kStages;
        mbar_wait(&full[sl], (last / kStages) & 1, err, DFLASH_STATUS_TIMEOUT, nullptr);
      }
      if (has_block) mbar_wait(blk_full, 0, err, DFLASH_STATUS_TIMEOUT, nullptr);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ score MMA issuer
      constexpr uint32_t kIdS2 = idesc_bf16_f32(kRows, kSK);
      constexpr uint32_t kIdS1 = idesc_bf16_f32(kRows, kTK);
      constexpr uint32_t kIdSB = idesc_bf16_f32(kRows, kBK);
      bool ok = mbar_wait(q_tm, 0, err, DFLASH_STATUS_TIMEOUT, abort_word);
      bool any = false;
      // S_j = Q K_j^T once step j's keys have landed: one MMA per 16 dims,
      // 128 (or, for a last odd tile, 64) columns wide
      auto s_issue = [&](int j) -> bool {
        const bool blk = j == nsc;
        const int t0 = 2 * j;
        bool r;
        if (blk) {
          r = mbar_wait(blk_full, 0, err, DFLASH_STATUS_TIMEOUT, abort_word);
        } else {
          r = mbar_wait(&full[t0 % kStages], (t0 / kStages) & 1, err, DFLASH_STATUS_TIMEOUT, abort_word);
          if (r && t0 + 1 < nctx)
            r = mbar_wait(&full[(t0 + 1) % kStages], ((t0 + 1) / kStages) & 1, err, DFLASH_STATUS_TIMEOUT,
                          abort_word);
        }
        if (!r) return false;
        tc_fence_after();
        const uint32_t id = blk ? kIdSB : (t0 + 1 < nctx ? kIdS2 : kIdS1);
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t off = (kk & 3) * 32;
          const uint32_t kb = blk ? sbase + TcSmem::kBlock + (kk >> 2) * kBSub
                                  : sbase + (kk >= 4 ? TcSmem::kKhi : TcSmem::kKlo) + (t0 % kStages) * kSlot;
          umma_bf16_ta(tmem + kColS, tmem + kColQ + kk * 8, sdesc_sw128(kb + off), id, kk > 0 ? 1u : 0u);
        }
        umma_commit(s_full);
        return true;
      };
      if (ok && nS >= 1) {
        ok = s_issue(0);
        any = ok;
      }
      // the next step's scores as soon as softmax u has read this step's
      for (int u = 0; u + 1 < nS && ok; ++u) {
        ok = mbar_wait(s_empty, u & 1, err, DFLASH_STATUS_TIMEOUT, abort_word);
        if (ok) ok = s_issue(u + 1);
      }
      // every score MMA completes before tensor memory is released
      if (any) {
        umma_commit(&drain[0]);
        mbar_wait(&drain[0], 0, err, DFLASH_STATUS_TIMEOUT, nullptr);
      }
    }
  } else if (warp == 2) {
    if (lane == 0) {
      // ------------------------------------------------ output MMA issuer
      constexpr uint32_t kIdO = idesc_bf16_f32(kRows, kD) | kIdescBTransposed;
      bool ok = true;
      bool any = false;
      // O += P_u V_u once the softmax warps wrote P_u (and rescaled O)
      for (int u = 0; u < nS && ok; ++u) {
        ok = mbar_wait(&p_full[u & 1], (u >> 1) & 1, err, DFLASH_STATUS_TIMEOUT, abort_word);
        if (!ok) break;
        tc_fence_after();
        const bool blk = u == nsc;
        const int t0 = 2 * u;
        const int nks = blk ? kBK / 16 : (t0 + 1 < nctx ? kSK : kTK) / 16;
        const uint32_t pa = tmem + static_cast<uint32_t>(kColP + (u & 1) * 64);
        for (int kk = 0; kk < nks; ++kk) {
          const uint32_t vb = blk ? sbase + TcSmem::kBlock + 2 * kBSub + kk * 16 * 128
                                  : sbase + TcSmem::kVlo + ((t0 + (kk >> 2)) % kStages) * kSlot + (kk & 3) * 16 * 128;
          const uint32_t lbo = blk ? kBSub : kRing;  // V dims 0-63 -> 64-127
          umma_bf16_ta(tmem + kColO, pa + kk * 8, sdesc_sw128_mn(vb, lbo), kIdO, (u > 0 || kk > 0) ? 1u : 0u);
        }
        any = true;
        umma_commit(&o_full[u & 1]);
        if (!blk) {
          umma_commit(&empty[t0 % kStages]);
          if (t0 + 1 < nctx) umma_commit(&empty[(t0 + 1) % kStages]);
        }
      }
      // every output MMA completes before tensor memory is released
      if (any) {
        umma_commit(&drain[1]);
        mbar_wait(&drain[1], 0, err, DFLASH_STATUS_TIMEOUT, nullptr);
      }
    }
  }

  // ---------------------------------------------------- softmax (warps 3-18)
  const int q4 = warp & 3;                     // the lane quadrant this warp may access
  const int part = warp >= 3 ? (warp - 3) >> 2 : 0;  // which 32 keys of a step (and 32 output columns)
  const int r = q4 * 32 + lane;
  const uint32_t tl = tmem + (static_cast<uint32_t>(q4 * 32) << 16);
  float* xchg = reinterpret_cast<float*>(smem + TcSmem::kXchg);
  float* lpart = reinterpret_cast<float*>(smem + TcSmem::kLPart);
  float m = -INFINITY, l = 0.f;  // the maximum the probabilities use, and this warp's keys' sum
  bool done_all = false;         // the last step's P*V has landed
  if (warp >= 3 && q4 < nact) {
    const float sc = rsqrtf(static_cast<float>(kD)) * 1.4426950408889634f;
    const int key0 = part * 32;
    {
      // this warp's rows of Q, dims 32*part .. 32*part+31, into tensor memory
      uint32_t qv[16];
      if (r < rows) {
        const uint4* src = reinterpret_cast<const uint4*>(
            a.Q + (static_cast<int64_t>(si) * 16 + (r & 15)) * (a.nq * kD) + (kvh * G + (r >> 4)) * kD + key0);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint4 w = src[c];
          qv[4 * c] = w.x;
          qv[4 * c + 1] = w.y;
          qv[4 * c + 2] = w.z;
          qv[4 * c + 3] = w.w;
        }
      } else {
#pragma unroll
        for (int c = 0; c < 16; ++c) qv[c] = 0u;
      }
      tmem_st16u(tl + kColQ + part * 16, qv);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(q_tm);
    }
    // The four warps of a quadrant run every step and meet once a step at a
    // named barrier that also ORs their failure flags, so a wait that gives
    // up in one warp stops all four (never a warp alone at the barrier);
    // after a failure the steps only keep the barrier count.
    bool ok = true;
    for (int j = 0; j < nS; ++j) {
      const bool blk = j == nsc;
      const int nvalid = blk ? kBK : min(kSK, nkeys - j * kSK);
      const int nmine = max(0, min(32, nvalid - key0));  // valid keys of this warp
      // every wait's outcome is made warp-uniform: the tensor-memory loads
      // and stores after it are warp-collective
      if (ok) ok = mbar_wait(s_full, j & 1, err, DFLASH_STATUS_TIMEOUT, abort_word);
      ok = __all_sync(0xffffffffu, ok);
      float sv[32];
      if (ok) {
        tc_fence_after();
        uint32_t u[32];
        tmem_ld32_async(tl + kColS + key0, u);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) sv[i] = __uint_as_float(u[i]);
        tc_fence_before();
        mbar_arrive(s_empty);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) sv[i] = -INFINITY;
      }
      if (nmine < 32) {
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (i >= nmine) sv[i] = -INFINITY;
      }
      float t0 = sv[0], t1 = sv[1], t2 = sv[2], t3 = sv[3];
#pragma unroll
      for (int i = 4; i < 32; i += 4) {
        t0 = fmaxf(t0, sv[i]);
        t1 = fmaxf(t1, sv[i + 1]);
        t2 = fmaxf(t2, sv[i + 2]);
        t3 = fmaxf(t3, sv[i + 3]);
      }
      // the step's maximum over the quadrant's four warps (raw scores; the
      // scale is positive)
      {
        float* slot = xchg + ((q4 * kParts + part) * 2 + (j & 1)) * 32;
        slot[lane] = fmaxf(fmaxf(t0, t1), fmaxf(t2, t3));
        if (named_bar_or(1 + q4, 128, ok ? 0 : 1)) ok = false;
        float mx = -INFINITY;
#pragma unroll
        for (int p2 = 0; p2 < kParts; ++p2) mx = fmaxf(mx, xchg[((q4 * kParts + p2) * 2 + (j & 1)) * 32 + lane]);
        t0 = mx;
      }
      if (!ok) continue;
      const float tmax = t0 * sc;
      // P*V of step j-2, the last reader of this step's P buffer, must have
      // landed (o_full[b] completes once for each step using P buffer b;
      // the next of them needs this step's P, so the wait cannot fall two
      // phases behind). A rescale of the output also waits for P*V of j-1.
      if (j >= 2) ok = mbar_wait(&o_full[j & 1], ((j - 2) >> 1) & 1, err, DFLASH_STATUS_TIMEOUT, abort_word);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) continue;
      // a row needs a rescale when its step maximum passes the one in use by
      // more than the margin; the tensor-memory loads and stores are
      // warp-collective, so the warp rescales when any of its rows needs it
      // (alpha = 1 for the others). The four warps of a quadrant decide
      // alike: they hold the same rows and the same step maxima.
      const bool need = tmax > m + kRescaleLog2;
      const bool rescale = __any_sync(0xffffffffu, need);
      if (rescale) {
        if (j >= 1) ok = mbar_wait(&o_full[(j - 1) & 1], ((j - 1) >> 1) & 1, err, DFLASH_STATUS_TIMEOUT, abort_word);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) continue;
        tc_fence_after();
        const float alpha = !need ? 1.f : (m == -INFINITY ? 0.f : ex2(m - tmax));
        l *= alpha;
        if (j >= 1) {
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            float v[16];
            tmem_ld16(tl + kColO + part * 32 + c * 16, v);
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] *= alpha;
            tmem_st16(tl + kColO + part * 32 + c * 16, v);
          }
        }
        if (need) m = tmax;
      }
      const float negm = -m;
      float ps0 = 0.f, ps1 = 0.f, ps2 = 0.f, ps3 = 0.f;
#pragma unroll
      for (int i = 0; i < 32; i += 4) {
        sv[i] = ex2(fmaf(sv[i], sc, negm));
        sv[i + 1] = ex2(fmaf(sv[i + 1], sc, negm));
        sv[i + 2] = ex2(fmaf(sv[i + 2], sc, negm));
        sv[i + 3] = ex2(fmaf(sv[i + 3], sc, negm));
        ps0 += sv[i];
        ps1 += sv[i + 1];
        ps2 += sv[i + 2];
        ps3 += sv[i + 3];
      }
      l += (ps0 + ps1) + (ps2 + ps3);
      // this warp's keys of P as bf16 pairs into the step's P buffer
      {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const __nv_bfloat162 h = __floats2bfloat162_rn(sv[2 * e], sv[2 * e + 1]);
          pk[e] = *reinterpret_cast<const uint32_t*>(&h);
        }
        tmem_st16u(tl + kColP + (j & 1) * 64 + part * 16, pk);
        tmem_wait_st();
      }
      tc_fence_before();
      mbar_arrive(&p_full[j & 1]);
    }
    // the last P*V (its completion implies every earlier one)
    if (ok && nS >= 1)
      done_all = mbar_wait(&o_full[(nS - 1) & 1], ((nS - 1) >> 1) & 1, err, DFLASH_STATUS_TIMEOUT, abort_word);
    done_all = __all_sync(0xffffffffu, done_all);
    lpart[part * kRows + r] = l;
  }
  __syncthreads();  // every step consumed: the ring memory is free

  // this CTA's partial rows: part[r][kPartLd] (fp32) and ml[r][2]
  float* partial = reinterpret_cast<float*>(smem + TcSmem::kKlo);
  float* ml = partial + kRows * kPartLd;
  if (warp >= 3 && q4 < nact) {
    if (done_all) tc_fence_after();
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      float v[16];
      if (done_all) {
        tmem_ld16(tl + kColO + part * 32 + c * 16, v);
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = 0.f;
      }
      if (r < rows) {
        float4* pr = reinterpret_cast<float4*>(partial + r * kPartLd + part * 32 + c * 16);
#pragma unroll
        for (int i = 0; i < 4; ++i) pr[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
      }
    }
    if (r < rows && part == 0) {
      float lsum = 0.f;
#pragma unroll
      for (int p2 = 0; p2 < kParts; ++p2) lsum += lpart[p2 * kRows + r];
      ml[r * 2] = done_all ? m : -INFINITY;
      ml[r * 2 + 1] = done_all ? lsum : 0.f;
    }
  }
  csync();  // every CTA's partial is ready

  // reduce-scatter: this rank owns rows [v0, v1) of the 16*G
  {
    const int v0 = static_cast<int>(rank) * rows / CS;
    const int v1 = (static_cast<int>(rank) + 1) * rows / CS;
    const uint32_t pbase = smem_u32(partial), mlbase = smem_u32(ml);
    for (int idx = threadIdx.x; idx < (v1 - v0) * 32; idx += blockDim.x) {
      const int vec = v0 + idx / 32;
      const int d4 = (idx & 31) * 4;
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
      const int head = vec >> 4, row = vec & 15;
      __nv_bfloat16* out = a.out + (static_cast<int64_t>(si) * 16 + row) * (a.nq * kD) + (kvh * G + head) * kD + d4;
      const float inv = den > 0.f ? 1.f / den : 0.f;
      *reinterpret_cast<__nv_bfloat162*>(out) = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
      *reinterpret_cast<__nv_bfloat162*>(out + 2) = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
    }
  }
  csync();  // partials stay alive until every rank has read them
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
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

bool set_smem(void (*kern)(TcArgs)) {
  static std::mutex mu;
  static std::vector<void (*)(TcArgs)> done;
  std::lock_guard<std::mutex> lk(mu);
  for (auto k : done)
    if (k == kern) return true;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLaunch) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  done.push_back(kern);
  return true;
}

}  // namespace

bool attention_tc_supported(const AttnArgs& a) {
  const int G = a.nq / a.nkv;
  return a.d == kD && G >= 1 && G <= 8 && a.nq % a.nkv == 0;
}

int launch_attention_tc(const AttnArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap, int s_count,
                        int num_sms, cudaStream_t st) {
  static thread_local TcArgs P;
  P.a = a;
  P.kmap = kmap;
  P.vmap = vmap;
  const int T = s_count * 16;
  {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(a.nkv) * kD, static_cast<cuuint64_t>(T)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(a.nkv) * kD * 2};
    const cuuint32_t box[2] = {64, 16};
    int rc = encode_map(&P.kbmap, a.Kb, 2, dims, strides, box);
    if (!rc) rc = encode_map(&P.vbmap, a.Vb, 2, dims, strides, box);
    if (rc) return rc;
  }
  // keys a CTA: each (stream, kv head) splits over the most CTAs (a power
  // of two up to 8) whose grid still fits one wave of one CTA an SM; with
  // more (stream, kv head) pairs than SMs, one CTA each (a CTA's start and
  // merge cost about as much as eight key tiles, so fewer, longer CTAs win)
  const int units = s_count * a.nkv;
  int CS = 1;
  while (CS < 8 && units * CS * 2 <= num_sms) CS *= 2;
  void (*kern)(TcArgs) = CS == 1 ? attn_tc_kernel<1> : CS == 2 ? attn_tc_kernel<2> : CS == 4 ? attn_tc_kernel<4>
                                                                                             : attn_tc_kernel<8>;
  if (!set_smem(kern)) return DFLASH_E_CUDA;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(CS);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(CS), a.nkv, s_count);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemLaunch;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  TraceScope ts(st, "attention", a.trace_bytes, 0.0);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, P);
  count_launch();
  return cuda_status(e);
}

}  // namespace dfl
