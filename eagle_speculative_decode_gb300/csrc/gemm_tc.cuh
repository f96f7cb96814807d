#pragma once
// Tensor-core (tcgen05) GEMM for the drafter's projections at batched sizes: the rows of
// a weight matrix against N activation rows (items) at once, so each weight byte is read
// from HBM once for the whole batch.
//
// y[item, row] = sum_k W[row, k] * x[item, k].  The MMA's M side is 128 weight rows, its N
// side the items (16..128), K in 64-element k-tiles ("swap AB": the weights are the A
// operand, the activations the B operand; both K-major in shared memory, 128-byte
// swizzled, loaded by TMA).  float32 activations are split into three bf16 parts
// x = x0 + x1 + x2 (exact to float32's 24 bits) and every part is multiplied; bf16
// features (the encode) are one part.
//
// Two schedules, one CTA per SM:
//  * cluster split-K, when there are few tiles (T <= 76): each tile gets s CTAs
//    (2 <= s <= 8, T * s at least 60% of the SM count) in one thread-block cluster, each
//    multiplying a contiguous 1/s of K.  The s float32 partial tiles meet in distributed
//    shared memory: after one cluster barrier every rank adds, for its own share of the
//    item columns, the s partials in rank order and runs the tile epilogue on those
//    columns, so neither the reduction nor the epilogue waits on one CTA.
//  * persistent stream-K otherwise: every CTA walks an equal share of all (tile, k-tile)
//    units, tile by tile, so no SM idles in a tail wave.  A tile that two or more CTAs
//    share is finished by the last of them, which adds the others' float32 partial sums
//    (published through L2) in CTA order.
//
// The three parts sit on consecutive rows of the B tile, so one MMA of width 3N multiplies
// them all (the x0, x1, x2 products land in adjacent TMEM column blocks).  Precision: a
// TMEM accumulator takes at most kTcChunk k-tiles (4 * kTcChunk MMAs), then the epilogue
// warps add the chunk into float32 registers; two TMEM buffers alternate, so the MMAs do
// not wait for the drain.
//
// Warp roles (352 threads): warps 0-7 drain TMEM and run the fused epilogues (two warps
// per TMEM lane quadrant), warp 8 streams the weight tiles (deep ring: the HBM stream),
// warp 9 issues the MMAs (one thread) and owns TMEM, warp 10 streams the activation
// tiles (shallow ring: they come from L2); with INT4 weights warp 8 streams code tiles
// and warps 11-14 decode them into the weight ring.  Every mbarrier wait is bounded
// (EAGLE3_DEV_TIMEOUT), and no copy is left in flight when the CTA finishes.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "epilogue.cuh"
#include "internal.h"

namespace e3 {

constexpr int kTcM = 128;          // MMA M (weight rows per tile)
constexpr int kTcK = 64;           // k-tile: one 128-byte swizzle row of bf16
constexpr int kTcAWarp = 8, kTcMmaWarp = 9, kTcBWarp = 10;
constexpr int kTcThreads = 352;
// INT4 weights: four more warps (11-14) decode the code tiles into the weight ring
constexpr int kTcConvWarp0 = 11, kTcConvWarps = 4;
constexpr int kTcThreadsQ4 = kTcThreads + 32 * kTcConvWarps;
constexpr int kTcChunk = 8;        // k-tiles per TMEM accumulation chunk
constexpr int kTcEpiThreads = 256; // warps 0-7: TMEM drain and epilogues

// Barrier among the 256 epilogue threads (the producer and MMA warps are not in it).
__device__ __forceinline__ void tc_epi_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

struct TcArgs {
  CUtensorMap a0;   // weight matrix of the tile (q / fc / o / gate / down / lm_head)
  CUtensorMap a1;   // second matrix: k (q/k/v) or up (gate/up)
  CUtensorMap a2;   // third matrix: v (q/k/v)
  CUtensorMap b0;   // activations [M, K] bf16: the bf16 features, or x0 of the split
  CUtensorMap b1;   // x1 of the split
  CUtensorMap b2;   // x2 of the split
  GemvParams p;     // epilogue parameters (p.items = M, p.item0 = 0)
  const uint32_t *sz0, *sz1, *sz2;  // INT4: (scale, zero) rows of the a0 / a1 / a2 codes
  int sz_stride;                    // INT4: pairs per (scale, zero) row
  const float *gsum;                // INT4: [M][K / 128] sum of x over each 128-wide group
  const float *sumsq;  // [M][halves] sum of squares of the staged x (norm modes)
  float *part;         // stream-K partials [grid][2][N][128]
  unsigned *tile_cnt;  // stream-K arrival counters [tiles], zero between launches
  int csplit;          // cluster split-K: CTAs per tile (= cluster size); 0: stream-K
  int M;               // items in total
  int item_tiles, row_tiles, ktiles;
  int units;           // tiles * ktiles
};

// ------------------------------------------------------------------ PTX helpers
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, 8-row atoms of
// 1024 bytes (stride byte offset), descriptor version 1.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);   // start address
  d |= (uint64_t)1 << 16;                     // leading byte offset (unused for swizzled K-major)
  d |= (uint64_t)(1024 >> 4) << 32;           // stride byte offset
  d |= (uint64_t)1 << 46;                     // version
  d |= (uint64_t)2 << 61;                     // layout: 128-byte swizzle
  return d;
}

// Instruction descriptor of kind::f16: bf16 A and B, float32 accumulate, both K-major.
__host__ __device__ constexpr uint32_t tc_idesc(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void tc_mma(uint32_t dtmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(dtmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The same with the A operand in tensor memory (128 lanes = rows, K packed two bf16 to a
// 32-bit column, the even k in the low half).
__device__ __forceinline__ void tc_mma_ta(uint32_t dtmem, uint32_t atmem, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(dtmem),
      "r"(atmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 16 consecutive float32 columns of this thread's TMEM lane, added into acc.
__device__ __forceinline__ void tmem_add16(uint32_t taddr, float *acc) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] += __uint_as_float(r[i]);
}

// 32 consecutive 32-bit columns of this thread's TMEM lane, written and waited for.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
      "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
      "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 16 consecutive 32-bit columns of this thread's TMEM lane, loaded without waiting (the
// caller waits once for several loads with tmem_wait_ld).
__device__ __forceinline__ void tmem_ld16_async(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 16 consecutive float32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float *v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// INT4 codes of one 32-bit word (byte j: input 2j in the low nibble, 2j + 1 in the high
// one) as 8 bf16 weights code - 8, in input order.  A code c becomes the bf16 128 + c (the
// exponent of 128, c in the low mantissa bits) by a byte permute and a mask; one packed
// subtraction of 136 then gives c - 8, exactly (both operands and the difference are
// representable).
__device__ __forceinline__ uint4 q4_to_bf16x8(uint32_t w) {
  const uint32_t t = w & 0x0F0F0F0Fu, u = (w >> 4) & 0x0F0F0F0Fu;  // even / odd inputs
  uint32_t o[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t v = (__byte_perm(t, u, 0x4400u + 0x1111u * q) & 0x000F000Fu) | 0x43004300u;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(o[q]) : "r"(v), "r"(0x43084308u));
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// ------------------------------------------------------------------ shapes
template <int MODE>
struct TcMode {
  static constexpr int H = ModeTraits<MODE>::kHalves;
  static constexpr int P = MODE == GM_ENCODE ? 1 : 3;  // bf16 parts of x
  static constexpr int kMaxN = MODE == GM_ENCODE ? 128 : 64;
  static constexpr bool kStaging = MODE == GM_QKV || MODE == GM_GATEUP;  // row exchange
};

template <int N, int MODE, bool Q4 = false>
struct TcShape {
  using T = TcMode<MODE>;
  static constexpr int H = T::H, P = T::P;
  static constexpr int kA = kTcM * kTcK * 2;            // 16 KB bf16 weight tile
  static constexpr int kAS = Q4 ? 0 : kA;                // its shared-memory ring slot (INT4: in TMEM)
  static constexpr int kQ = Q4 ? kTcM * kTcK / 2 : 0;   // INT4: 4 KB of codes per k-tile
  static constexpr int kB = N * kTcK * 2;               // one activation part
  static constexpr int kBStage = P * kB;
  // TMEM: chunk buffers of [P][N] columns (a chunk lies in one K half), used in turn: two
  // for bf16 weights (chunks of 8 k-tiles); INT4 drains every group (2 k-tiles), so it
  // takes as many as fit in 384 columns, up to 8, to let the MMAs run ahead of the drains
  static constexpr int NP = P * N;                      // MMA width: the parts stacked
  static_assert(NP % 16 == 0 && NP <= 256, "MMA N of kind::f16 with M = 128");
  static constexpr int NBUF = Q4 ? (384 / NP >= 8 ? 8 : (384 / NP >= 4 ? 4 : 2)) : 2;
  // INT4: the decoded weight tiles live in TMEM too, 32 columns (64 k of bf16) per stage
  // after the accumulators
  static constexpr int kACol0 = NBUF * NP;
  static constexpr int kCols = NBUF * NP + (Q4 ? 4 * 32 : 0);
  static_assert(kCols <= 512, "accumulators fit in TMEM");
  static constexpr int kTmemCols = kCols <= 32 ? 32 : kCols <= 64 ? 64 : kCols <= 128 ? 128 : kCols <= 256 ? 256 : 512;
  static constexpr int NCH = N >= 32 ? N / 32 : 1;      // 16-column chunks per epilogue thread
  static constexpr int kStageBytes = T::kStaging ? kTcM * (N + 1) * 4 : 0;
  // lm_head: per-quad best keys of a tile [4][N] and the CTA's running best [N] (u64)
  static constexpr int kLmBytes = MODE == GM_LMHEAD ? 5 * N * 8 : 0;
  // INT4: the items' sums of x over the groups of the current segment, [group][N] floats
  static constexpr int kQsumFloats = Q4 ? 2048 : 0;
  static constexpr int kAux = 3072;                      // barriers and per-item tables
  // activation ring: shallow for bf16 weights (L2 hits; the weight ring, the HBM stream,
  // takes the rest).  INT4 streams 4 KB of codes per k-tile, so the activations' L2
  // latency sets the pace unless their ring is deep: 96 KB of activation tiles.
  static constexpr int kNB = Q4 ? (96 * 1024 / kBStage > 16 ? 16 : 96 * 1024 / kBStage) : (kBStage <= 12 * 1024 ? 4 : 3);
  static constexpr int kFixed = 1024 /*alignment*/ + kAux + kStageBytes + kLmBytes + 4 * kQsumFloats + kNB * kBStage;
  // bf16: the weight ring takes the rest (at most 12 stages).  INT4: four TMEM stages of
  // decoded tiles, and the codes' ring (the HBM stream) takes the rest (at most 32 stages).
  static constexpr int kFitA = (int)((kTcSmemLimit - kFixed) / kA);
  static constexpr int kNA = Q4 ? 4 : (kFitA > 12 ? 12 : kFitA);  // weight (decoded) ring stages
  static_assert((Q4 || kFitA >= kNA) && kNA >= 4, "a weight ring of four stages");
  static constexpr int kFitQ = Q4 ? (int)((kTcSmemLimit - kFixed - kNA * kAS) / (kQ > 0 ? kQ : 1)) : 0;
  static constexpr int kNQ = kFitQ > 32 ? 32 : kFitQ;   // INT4 code ring stages
  static_assert(!Q4 || kNQ >= 4, "an INT4 code ring of four stages");
  // a tile's float32 partial sums fit the idle rings (cluster exchange, stream-K fix-up)
  static_assert((size_t)N * kTcM * 4 <= (size_t)kNA * kAS + (size_t)kNB * kBStage, "partials fit the rings");
  static constexpr int kSmem = kFixed + kNA * kAS + kNQ * kQ;
  static __device__ __forceinline__ uint32_t buf_col(int b) { return (uint32_t)(b * NP); }
};

// The partition: CTA c owns units [start(c), start(c + 1)) of the flattened
// (tile, k-tile) space, tiles ordered row tile major, item tile minor.  Stream-K cuts it
// into equal shares; cluster split-K gives rank q of tile t's cluster the k-tiles
// [q * ktiles / s, (q + 1) * ktiles / s) of that tile.
struct TcSched {
  int units, grid, ktiles, csplit;
  __host__ __device__ int start(int c) const {
    if (csplit > 0) {
      const int t = c / csplit, q = c - t * csplit;
      return t * ktiles + (ktiles * q) / csplit;
    }
    return (int)(((long long)units * c) / grid);
  }
  __host__ __device__ int cta_of(int u) const {
    int c = (int)(((long long)u * grid) / units);
    while (c + 1 < grid && start(c + 1) <= u) ++c;
    while (c > 0 && start(c) > u) --c;
    return c;
  }
};

// One contiguous run of k-tiles [kt0, kt1) of tile t inside a CTA's share.
struct TcSeg {
  int t, kt0, kt1;
};

__device__ __forceinline__ TcSeg tc_seg(int u, int uend, int ktiles) {
  TcSeg s;
  s.t = u / ktiles;
  s.kt0 = u - s.t * ktiles;
  s.kt1 = min(ktiles, s.kt0 + (uend - u));
  return s;
}

// K half (q/k/v: [embed ; g], normalised separately) of k-tile kt.
template <int H>
__device__ __forceinline__ int tc_half(int kt, int n_embd) {
  return (H == 2 && kt * kTcK >= n_embd) ? 1 : 0;
}

// End of the accumulation chunk that starts at k-tile cb inside a segment ending at kt1:
// chunks end at multiples of kTcChunk and at the K half boundary (nh_tiles), so each
// chunk lies in one half.
template <int H, int CHK = kTcChunk>
__device__ __forceinline__ int tc_chunk_end(int cb, int kt1, int nh_tiles) {
  int ce = min(kt1, (cb / CHK + 1) * CHK);
  if (H == 2 && cb < nh_tiles && ce > nh_tiles) ce = nh_tiles;
  return ce;
}

// ------------------------------------------------------------------ cluster helpers
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Every thread of every CTA of the cluster (no .aligned form: threads may arrive apart).
// Each thread reaches the kernel's cluster barriers on every path, so the wait ends.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
// Address of the same shared-memory location in cluster rank `rank`.
__device__ __forceinline__ uint32_t dsmem_map(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ float ld_dsmem(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

// One lane of the (converged) warp, the same lane every time for the same mask.
__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n .reg .pred P;\n elect.sync _|P, 0xffffffff;\n selp.u32 %0, 1, 0, P;\n}\n"
      : "=r"(pred));
  return pred != 0;
}

// mbar_wait on every lane of the warp; true only when all lanes saw the phase, so the warp
// leaves converged.
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag, int *status) {
  if (__all_sync(0xffffffffu, mbar_test(bar, parity))) return true;  // the usual case: already there
  const bool ok = mbar_wait(bar, parity, abort_flag, status);
  return __all_sync(0xffffffffu, ok) != 0;
}

// Wait without the CTA's abort shortcut (still bounded): used to drain copies and MMAs
// that are in flight before the CTA releases its shared memory and TMEM.
__device__ __forceinline__ void tc_drain_wait(uint32_t bar, uint32_t parity) {
  for (uint32_t i = 0; i < kWaitLimit; ++i) {
    if (mbar_try_wait(bar, parity)) return;
    if (i > 64) __nanosleep(64);
  }
}

// ------------------------------------------------------------------ tile epilogues
// Thread (quad, chalf, lane) holds TMEM lane r = 32 * quad + lane (row r of the tile) and
// the 16-column chunks c0(j) = (2 j + chalf) * 16 < N (items item0 + c0(j) + i).
template <int N>
__device__ __forceinline__ int tc_c0(int j, int chalf) {
  return N >= 32 ? (2 * j + chalf) * 16 : 0;
}
template <int N>
__device__ __forceinline__ bool tc_has(int j, int chalf) {
  return N >= 32 ? true : chalf == 0;
}

struct TcTables {
  float *scale;  // [N][H] RMSNorm scales of the tile's items
  int *pos;      // [N] q/k/v: position, sequence and keep flag of each item
  int *seq;
  int *keep;
  int *page;     // [N] q/k/v: physical KV page of each kept item's position (-1: none)
  float *stage;  // [128][N + 1] row exchange (q/k/v RoPE partners, gate/up)
  unsigned long long *quad_best;  // lm_head [4][N]
  unsigned long long *run_best;   // lm_head [N]: this CTA's best so far, item tile run_it
};

// Max of NV 64-bit keys per lane across the warp, transposed: afterwards lane l holds the
// maximum of value index warp_reduce_index<NV>(l) (writers: warp_reduce_writer<NV>(l)).
template <int NV>
__device__ __forceinline__ unsigned long long warp_max_multi(unsigned long long (&v)[NV], int lane) {
  static_assert(NV >= 1 && NV <= 32 && (NV & (NV - 1)) == 0, "1..32 values, a power of two");
#pragma unroll
  for (int cnt = NV, o = 16; cnt > 1; cnt >>= 1, o >>= 1) {
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < cnt / 2; ++i) {
      const unsigned long long send = upper ? v[i] : v[i + cnt / 2];
      const unsigned long long keep = upper ? v[i + cnt / 2] : v[i];
      const unsigned long long other = __shfl_xor_sync(0xffffffffu, send, o);
      v[i] = keep > other ? keep : other;
    }
  }
  unsigned long long r = v[0];
#pragma unroll
  for (int o = 16 >> Log2<NV>::value; o >= 1; o >>= 1) {
    const unsigned long long other = __shfl_xor_sync(0xffffffffu, r, o);
    r = other > r ? other : r;
  }
  return r;
}

// lm_head: push the CTA's running best keys (item tile it) to the global argmax slots.
template <int N>
__device__ __forceinline__ void tc_lm_flush(const TcArgs &A, const TcTables &tb, int it) {
  const int tid = threadIdx.x;
  if (tid < N) {
    const unsigned long long k = tb.run_best[tid];
    const int item = it * N + tid;
    if (k != 0ull && item < A.M) atomicMax(A.p.am_slot + item, k);
    tb.run_best[tid] = 0ull;
  }
}

// INT4: the (scale, zero) row of tile row r of row tile rt (null past the matrix's end).
template <int MODE>
__device__ __forceinline__ const uint32_t *tc_q4_sz_row(const TcArgs &A, int rt, int r) {
  const GemvParams &p = A.p;
  if constexpr (MODE == GM_QKV) {
    const int qr = p.n_head * p.head_dim, kr = p.n_head_kv * p.head_dim;
    const int lr = p.row_base + rt * kTcM + r;
    if (lr < qr) return A.sz0 + (size_t)lr * A.sz_stride;
    if (lr < qr + kr) return A.sz1 + (size_t)(lr - qr) * A.sz_stride;
    if (lr < qr + 2 * kr) return A.sz2 + (size_t)(lr - qr - kr) * A.sz_stride;
    return nullptr;
  } else if constexpr (MODE == GM_GATEUP) {
    const int row = rt * 64 + (r & 63);  // tile rows 0-63 gate, 64-127 the matching up rows
    if (row >= p.n_ff) return nullptr;
    return (r < 64 ? A.sz0 : A.sz1) + (size_t)row * A.sz_stride;
  } else {
    const int row = rt * kTcM + r;
    return row < p.rows ? A.sz0 + (size_t)row * A.sz_stride : nullptr;
  }
}

// Per-item tables of item tile it: RMSNorm scales and, for q/k/v, each item's position,
// sequence, keep flag and KV page (status bits for a bad position or page of a kept item).
// Run by the epilogue warps while the MMAs of the CTA's first chunks are in flight.
template <int N, int MODE>
__device__ void tc_tables(const TcArgs &A, int it, const TcTables &tb) {
  constexpr int H = TcShape<N, MODE>::H;
  const GemvParams &p = A.p;
  const int tid = threadIdx.x;
  const int item0 = it * N;
  if constexpr (ModeTraits<MODE>::kNorm) {
    for (int i = tid; i < N * H; i += kTcEpiThreads) {
      const int c = i / H, h = i - c * H, item = item0 + c;
      tb.scale[i] = item < A.M ? rsqrtf(A.sumsq[(size_t)item * H + h] / (float)(p.K / H) + p.eps) : 0.f;
    }
  }
  if constexpr (MODE == GM_QKV) {
    // each kept item's KV page, looked up once per item
    for (int c = tid; c < N; c += kTcEpiThreads) {
      const int item = item0 + c;
      int pos = 0, seq = 0, keep = 0, page = -1;
      if (item < A.M) {
        const PairItem pi = resolve_pair(p.pairs, item, p.n_embd);
        pos = pi.pos;
        seq = pi.b;
        keep = pi.write_kv ? 1 : 0;
        if (keep) {
          if (pos < 0 || pos >= p.max_cache_len) {
            set_status(p.status, EAGLE3_DEV_BAD_POSITION);
          } else {
            page = p.page_table[(size_t)seq * p.max_pages + pos / p.page_size];
            if (page < 0 || page >= p.num_pages) {
              set_status(p.status, EAGLE3_DEV_BAD_PAGE);
              page = -1;
            }
          }
        }
      }
      tb.pos[c] = pos;
      tb.seq[c] = seq;
      tb.keep[c] = keep;
      tb.page[c] = page;
    }
  }
}

template <int N, int MODE>
__device__ void tc_tile_epilogue(const TcArgs &A, float (&acc)[TcShape<N, MODE>::H][TcShape<N, MODE>::NCH][16],
                                 int rt, int it, const TcTables &tb, unsigned ownm) {
  using S = TcShape<N, MODE>;
  constexpr int H = S::H, NCH = S::NCH, SP = N + 1;
  const GemvParams &p = A.p;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int quad = warp & 3, chalf = warp >> 2, r = quad * 32 + lane;
  const int item0 = it * N;
  // chunk j of this thread is written by this CTA (cluster split-K: its share of the columns)
  auto own = [&](int j) { return tc_has<N>(j, chalf) && ((ownm >> j) & 1u); };

  // y: the tile's sums, the K halves already scaled by their RMSNorm factors and added
  float(&y)[NCH][16] = acc[0];

  if constexpr (MODE == GM_ENCODE || MODE == GM_O || MODE == GM_DOWN) {
    const int row = rt * kTcM + r;
    if (row < p.rows) {
      // all residual loads first (independent, in flight together), then the stores
      if constexpr (MODE != GM_ENCODE) {
#pragma unroll
        for (int j = 0; j < NCH; ++j) {
          if (!own(j)) continue;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int item = item0 + tc_c0<N>(j, chalf) + i;
            if (item < A.M) y[j][i] += __ldcg(p.res + (size_t)item * p.rows + row);
          }
        }
      }
#pragma unroll
      for (int j = 0; j < NCH; ++j) {
        if (!own(j)) continue;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int item = item0 + tc_c0<N>(j, chalf) + i;
          if (item >= A.M) continue;
          p.out_f[(size_t)item * p.rows + row] = y[j][i];
          if constexpr (MODE == GM_DOWN) {
            if (p.dbg_f) p.dbg_f[(size_t)item * p.dbg_stride_b + p.dbg_off + row] = y[j][i];
          }
        }
      }
    }
  } else if constexpr (MODE == GM_LMHEAD) {
    // per item: best (logit, lowest row) of the warp's 32 rows by a transposed shuffle
    // reduction, then of the 4 lane quadrants in shared memory, folded into the CTA's
    // running best (pushed to the global slots once per item tile).
    constexpr int NV = NCH * 16;
    const int row = rt * kTcM + r;
    const bool vrow = row < p.rows;
    if (tc_has<N>(0, chalf)) {
      unsigned long long keys[NV];
#pragma unroll
      for (int j = 0; j < NCH; ++j)
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int item = item0 + tc_c0<N>(j, chalf) + i;
          const float v = y[j][i];
          const bool ok = vrow && own(j);
          if (ok && item < A.M && p.dbg_f) p.dbg_f[(size_t)item * p.dbg_stride_b + p.dbg_off + row] = v;
          keys[j * 16 + i] = ok ? (((unsigned long long)float_order_key(v) << 32) |
                                     (unsigned long long)(0xFFFFFFFFu - (uint32_t)row))
                                  : 0ull;
        }
      const unsigned long long best = warp_max_multi<NV>(keys, lane);
      if (warp_reduce_writer<NV>(lane)) {
        const int vi = warp_reduce_index<NV>(lane);
        tb.quad_best[quad * N + tc_c0<N>(vi / 16, chalf) + (vi % 16)] = best;
      }
    }
    tc_epi_sync();
    if (tid < N) {
      unsigned long long b = tb.run_best[tid];
#pragma unroll
      for (int q = 0; q < 4; ++q) b = tb.quad_best[q * N + tid] > b ? tb.quad_best[q * N + tid] : b;
      tb.run_best[tid] = b;
    }
    tc_epi_sync();
    if (A.item_tiles > 1) {  // the next tile may belong to another item tile
      tc_lm_flush<N>(A, tb, it);
      tc_epi_sync();
    }
  } else if constexpr (MODE == GM_GATEUP) {
    // tile rt: gate rows rt*64 + i in tile rows i < 64, the matching up rows in 64 + i
    if (r >= 64) {
#pragma unroll
      for (int j = 0; j < NCH; ++j)
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (tc_has<N>(j, chalf)) tb.stage[(r - 64) * SP + tc_c0<N>(j, chalf) + i] = y[j][i];
    }
    tc_epi_sync();
    const int row = rt * 64 + r;
    if (r < 64 && row < p.n_ff) {
#pragma unroll
      for (int j = 0; j < NCH; ++j) {
        if (!own(j)) continue;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int c = tc_c0<N>(j, chalf) + i, item = item0 + c;
          if (item >= A.M) continue;
          p.out_f[(size_t)item * p.n_ff + row] = silu_f(y[j][i]) * tb.stage[r * SP + c];
        }
      }
    }
    tc_epi_sync();  // the staging area is free again
  } else if constexpr (MODE == GM_QKV) {
    const int d = p.head_dim, R = p.rope_dims, half = R >> 1;
    const int qr = p.n_head * d, kr = p.n_head_kv * d;
    const int lr0 = p.row_base + rt * kTcM;  // row of [q; k; v] at tile row 0
    const int region = lr0 < qr ? 0 : (lr0 < qr + kr ? 1 : 2);
    const int rr = lr0 + r - (region == 0 ? 0 : (region == 1 ? qr : qr + kr));
    const int head = rr / d, hr = rr - head * d;
    const bool rope = region < 2 && hr < R;
    const int rp = r + (hr < half ? half : -half);  // RoPE partner (same tile)
    const bool vrow = lr0 + r < qr + 2 * kr;
#pragma unroll
    for (int j = 0; j < NCH; ++j)
#pragma unroll
      for (int i = 0; i < 16; ++i)
        if (tc_has<N>(j, chalf)) tb.stage[r * SP + tc_c0<N>(j, chalf) + i] = y[j][i];
    tc_epi_sync();
    if (vrow) {
      // RoPE in registers first (partner from the staging area, angles from the table),
      // then the stores
      if (rope) {
        const int i0 = hr < half ? hr : hr - half;
#pragma unroll
        for (int j = 0; j < NCH; ++j) {
          if (!own(j)) continue;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int c = tc_c0<N>(j, chalf) + i;
            const int pos = tb.pos[c];
            const int pr = (pos < 0 || pos >= p.max_cache_len) ? 0 : pos;
            const float2 cs = __ldg(p.rope + (size_t)pr * half + i0);
            const float pv = tb.stage[rp * SP + c];
            y[j][i] = hr < half ? y[j][i] * cs.x - pv * cs.y : y[j][i] * cs.x + pv * cs.y;
          }
        }
      }
#pragma unroll
      for (int j = 0; j < NCH; ++j) {
        if (!own(j)) continue;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int c = tc_c0<N>(j, chalf) + i, item = item0 + c;
          if (item >= A.M) continue;
          if (region == 0) {
            p.out_f[(size_t)item * qr + rr] = y[j][i];
          } else if (p.kv_stage) {
            // quantized KV: float32 into the staging buffer, kv_quant writes the blocks
            if (tb.keep[c]) p.kv_stage[((size_t)item * 2 + (region - 1)) * kr + rr] = y[j][i];
          } else {
            const int pg = tb.page[c];
            if (pg < 0) continue;
            const int pos = tb.pos[c];
            uint16_t *pool = region == 1 ? p.k_pool : p.v_pool;
            pool[(((size_t)pg * p.n_head_kv + head) * p.page_size + pos % p.page_size) * d + hr] = f2bf(y[j][i]);
          }
        }
      }
    }
    tc_epi_sync();  // the staging area is free again
  }
}

// ------------------------------------------------------------------ kernel
template <int N, int MODE, bool Q4>
__global__ void __launch_bounds__(Q4 ? kTcThreadsQ4 : kTcThreads, 1) gemm_tc_kernel(const __grid_constant__ TcArgs args) {
  using S = TcShape<N, MODE, Q4>;
  constexpr int H = S::H, P = S::P, NA = S::kNA, NB = S::kNB, NCH = S::NCH, NQ = S::kNQ;
  // k-tiles per TMEM accumulation chunk: INT4 drains every 128-wide group (two k-tiles)
  // to apply the group's scale
  constexpr int CHK = Q4 ? 2 : kTcChunk;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  // [A ring NA x 16 KB][B ring NB x P parts][INT4 code ring NQ x 4 KB][staging]
  // [barriers, flags, per-item tables]
  unsigned char *aring = smem;
  unsigned char *bring = aring + (size_t)NA * S::kAS;
  unsigned char *qring = bring + (size_t)NB * S::kBStage;
  float *stage = reinterpret_cast<float *>(qring + (size_t)NQ * S::kQ);
  unsigned char *lmb = reinterpret_cast<unsigned char *>(stage) + S::kStageBytes;
  float *qsum = reinterpret_cast<float *>(lmb + S::kLmBytes);  // INT4 group sums of the segment
  unsigned char *aux = reinterpret_cast<unsigned char *>(qsum + S::kQsumFloats);
  const uint32_t fullA = smem_addr(aux), emptyA = fullA + 8 * NA;
  const uint32_t fullB = emptyA + 8 * NA;
  constexpr int NBUF = S::NBUF;
  const uint32_t emptyB = fullB + 8 * NB;  // activation slot free (its MMAs' commit)
  const uint32_t hi_full = emptyB + 8 * NB, hi_free = hi_full + 8 * NBUF;
  const uint32_t mma_done = hi_free + 8 * NBUF;
  const uint32_t fix_bar = mma_done + 8;  // bulk copies of published partials (last tile)
  const uint32_t fullQ = fix_bar + 8, emptyQ = fullQ + 8 * NQ;  // INT4 code ring
  unsigned char *aux2 = aux + 8 * (2 * NA + 2 * NB + 2 * NBUF + 3 + 2 * NQ);
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(aux2);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(aux2 + 4);
  int *last_sh = reinterpret_cast<int *>(aux2 + 8);
  TcTables tb;
  tb.scale = reinterpret_cast<float *>(aux2 + 16);
  tb.pos = reinterpret_cast<int *>(tb.scale + N * H);
  tb.seq = tb.pos + N;
  tb.keep = tb.seq + N;
  tb.page = tb.keep + N;
  tb.stage = stage;
  tb.quad_best = reinterpret_cast<unsigned long long *>(lmb);
  tb.run_best = tb.quad_best + 4 * N;
  static_assert(8 * (2 * S::kNA + 2 * S::kNB + 2 * S::NBUF + 3 + 2 * S::kNQ) + 16 + 4 * (N * S::H + 4 * N) <= S::kAux, "aux area");

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const GemvParams &pc = args.p;
  const int ktiles = args.ktiles, item_tiles = args.item_tiles;
  TcSched sched;
  sched.units = args.units;
  sched.grid = gridDim.x;
  sched.ktiles = args.ktiles;
  sched.csplit = args.csplit;
  const int cta = blockIdx.x;
  const int u_begin = sched.start(cta), u_end = sched.start(cta + 1);

  if (warp == kTcMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_holder)),
                 "r"(S::kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 0) {
    for (int i = 0; i < NA; ++i) {
      mbar_init(fullA + 8 * i, Q4 ? kTcConvWarps : 1);  // INT4: one arrival per decoding warp
      mbar_init(emptyA + 8 * i, 1);
    }
    for (int i = 0; i < NQ; ++i) {
      mbar_init(fullQ + 8 * i, 1);
      mbar_init(emptyQ + 8 * i, kTcConvWarps);
    }
    for (int i = 0; i < NB; ++i) {
      mbar_init(fullB + 8 * i, 1);
      mbar_init(emptyB + 8 * i, 1);
    }
    for (int i = 0; i < NBUF; ++i) {
      mbar_init(hi_full + 8 * i, 1);
      mbar_init(hi_free + 8 * i, 8);  // one arrival per epilogue warp
    }
    mbar_init(mma_done, 1);
    mbar_init(fix_bar, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  pdl_trigger();

  // Producer and MMA warps run their loops with all 32 lanes converged (waits on every
  // lane, operands warp-uniform); one elected lane issues the copies, MMAs and commits.
  if (warp == kTcAWarp) {
    // ------------------------------------------------------------ weight tiles (HBM)
    const bool leader = elect_one();
    if (leader) {
      tma_prefetch_map(&args.a0);
      if (MODE == GM_QKV || MODE == GM_GATEUP) tma_prefetch_map(&args.a1);
      if (MODE == GM_QKV) tma_prefetch_map(&args.a2);
    }
    const uint64_t pol_w = l2_evict_first_policy();
    const uint32_t abase = smem_addr(aring);
    int g = 0;
    bool ok = true;
    for (int u = u_begin; u < u_end && ok;) {
      const TcSeg sg = tc_seg(u, u_end, ktiles);
      const int rt = sg.t / item_tiles;
      const CUtensorMap *amap = &args.a0;
      int arow = rt * kTcM;
      if constexpr (MODE == GM_QKV) {
        const int qr = pc.n_head * pc.head_dim, kr = pc.n_head_kv * pc.head_dim;
        const int lr = pc.row_base + rt * kTcM;
        if (lr < qr) {
          arow = lr;
        } else if (lr < qr + kr) {
          amap = &args.a1;
          arow = lr - qr;
        } else {
          amap = &args.a2;
          arow = lr - qr - kr;
        }
      } else if constexpr (MODE == GM_GATEUP) {
        arow = rt * 64;
      }
      for (int kt = sg.kt0; kt < sg.kt1; ++kt, ++g) {
        if constexpr (Q4) {
          // INT4: the k-tile's codes (32 bytes of each row) into the code ring; the
          // epilogue warps decode them into the weight ring
          const int s = g % NQ;
          if (g >= NQ && !warp_wait(emptyQ + 8 * s, ((g / NQ) - 1) & 1, abort_flag, pc.status)) {
            ok = false;
            break;
          }
          if (leader) {
            const uint32_t dst = smem_addr(qring) + (uint32_t)(s * S::kQ);
            mbar_expect_tx(fullQ + 8 * s, (uint32_t)S::kQ);
            if constexpr (MODE == GM_GATEUP) {
              tma_load_2d(dst, &args.a0, kt * (kTcK / 2), arow, fullQ + 8 * s, pol_w);
              tma_load_2d(dst + S::kQ / 2, &args.a1, kt * (kTcK / 2), arow, fullQ + 8 * s, pol_w);
            } else {
              tma_load_2d(dst, amap, kt * (kTcK / 2), arow, fullQ + 8 * s, pol_w);
            }
          }
        } else {
          const int s = g % NA;
          if (g >= NA && !warp_wait(emptyA + 8 * s, ((g / NA) - 1) & 1, abort_flag, pc.status)) {
            ok = false;
            break;
          }
          if (leader) {
            const uint32_t dst = abase + (uint32_t)(s * S::kA);
            mbar_expect_tx(fullA + 8 * s, (uint32_t)S::kA);
            if constexpr (MODE == GM_GATEUP) {
              tma_load_2d(dst, &args.a0, kt * kTcK, arow, fullA + 8 * s, pol_w);
              tma_load_2d(dst + S::kA / 2, &args.a1, kt * kTcK, arow, fullA + 8 * s, pol_w);
            } else {
              tma_load_2d(dst, amap, kt * kTcK, arow, fullA + 8 * s, pol_w);
            }
          }
        }
        __syncwarp();
      }
      u += sg.kt1 - sg.kt0;
    }
    if constexpr (Q4) {
      for (int q = max(0, g - NQ); q < g; ++q) tc_drain_wait(fullQ + 8 * (q % NQ), (q / NQ) & 1);
    } else {
      for (int q = max(0, g - NA); q < g; ++q) tc_drain_wait(fullA + 8 * (q % NA), (q / NA) & 1);
    }
    __syncwarp();
    if (args.csplit) cluster_sync_all();  // the epilogue warps' partial exchange
  } else if (warp == kTcBWarp) {
    // ------------------------------------------------------------ activation tiles (L2)
    const bool leader = elect_one();
    if (leader) tma_prefetch_map(&args.b0);
    uint64_t pol_x;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol_x));
    const uint32_t bbase = smem_addr(bring);
    pdl_wait();  // the activations come from the previous kernel
    int g = 0;
    bool ok = true;
    for (int u = u_begin; u < u_end && ok;) {
      const TcSeg sg = tc_seg(u, u_end, ktiles);
      const int ycoord = (sg.t % item_tiles) * N;
      for (int kt = sg.kt0; kt < sg.kt1; ++kt, ++g) {
        const int s = g % NB;
        // slot s last held stage g - NB: free once that stage's MMAs finished
        if (g >= NB && !warp_wait(emptyB + 8 * s, ((g / NB) - 1) & 1, abort_flag, pc.status)) {
          ok = false;
          break;
        }
        if (leader) {
          const uint32_t dst = bbase + (uint32_t)(s * S::kBStage);
          mbar_expect_tx(fullB + 8 * s, (uint32_t)S::kBStage);
          tma_load_2d(dst, &args.b0, kt * kTcK, ycoord, fullB + 8 * s, pol_x);
          if constexpr (P > 1) {
            tma_load_2d(dst + S::kB, &args.b1, kt * kTcK, ycoord, fullB + 8 * s, pol_x);
            tma_load_2d(dst + 2 * S::kB, &args.b2, kt * kTcK, ycoord, fullB + 8 * s, pol_x);
          }
        }
        __syncwarp();
      }
      u += sg.kt1 - sg.kt0;
    }
    for (int q = max(0, g - NB); q < g; ++q) tc_drain_wait(fullB + 8 * (q % NB), (q / NB) & 1);
    __syncwarp();
    if (args.csplit) cluster_sync_all();
  } else if (warp == kTcMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    const bool leader = elect_one();
    constexpr uint32_t idesc = tc_idesc(kTcM, S::NP);
    const int nh_tiles = pc.n_embd / kTcK;
    // descriptors of ring slot 0; slot s and K slice kk add (offset >> 4) to the start field
    const uint64_t adesc0 = smem_desc_sw128(smem_addr(aring));
    const uint64_t bdesc0 = smem_desc_sw128(smem_addr(bring));
    int g = 0, ch = 0;
    bool ok = true;
    for (int u = u_begin; u < u_end && ok;) {
      const TcSeg sg = tc_seg(u, u_end, ktiles);
      for (int cb = sg.kt0; cb < sg.kt1 && ok; ++ch) {
        const int ce = tc_chunk_end<H, CHK>(cb, sg.kt1, nh_tiles);
        const int hb = ch % NBUF;
        if (ch >= NBUF && !warp_wait(hi_free + 8 * hb, ((ch / NBUF) - 1) & 1, abort_flag, pc.status)) {
          ok = false;
          break;
        }
        const uint32_t dt = tmem + S::buf_col(hb);
        for (int kt = cb; kt < ce; ++kt, ++g) {
          const int sa = g % NA, sb = g % NB;
          if (!warp_wait(fullA + 8 * sa, (g / NA) & 1, abort_flag, pc.status) ||
              !warp_wait(fullB + 8 * sb, (g / NB) & 1, abort_flag, pc.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad0 = adesc0 + (uint64_t)((sa * S::kAS) >> 4);
          const uint64_t bd0 = bdesc0 + (uint64_t)((sb * S::kBStage) >> 4);
          if (leader) {
#pragma unroll
            for (int kk = 0; kk < kTcK / 16; ++kk) {  // 32 bytes further along K per slice
              if constexpr (Q4)  // decoded weights in TMEM: 8 columns per 16 k
                tc_mma_ta(dt, tmem + (uint32_t)(S::kACol0 + sa * 32 + kk * 8), bd0 + (uint64_t)(kk * 2), idesc,
                          (kt > cb || kk > 0) ? 1u : 0u);
              else
                tc_mma(dt, ad0 + (uint64_t)(kk * 2), bd0 + (uint64_t)(kk * 2), idesc, (kt > cb || kk > 0) ? 1u : 0u);
            }
            tc_commit(emptyA + 8 * sa);  // both rings' slots are free once these MMAs finish
            tc_commit(emptyB + 8 * sb);
          }
          __syncwarp();
        }
        if (ok) {
          if (leader) tc_commit(hi_full + 8 * hb);
          __syncwarp();
        }
        cb = ce;
      }
      u += sg.kt1 - sg.kt0;
    }
    // every MMA of this CTA has finished before TMEM is released
    if (leader) tc_commit(mma_done);
    __syncwarp();
    tc_drain_wait(mma_done, 0);
    __syncwarp();
    if (args.csplit) cluster_sync_all();
  } else if (Q4 && warp >= kTcConvWarp0) {
    // ------------------------------------------------------------ INT4 decoders
    // k-tile g of the CTA's share: its codes (code ring slot g % NQ) become bf16 weights
    // code - 8 in TMEM stage g % NA, as far ahead of the MMAs as the stages allow.  Warp w
    // owns TMEM lanes 32 (w % 4) .. +32 (a warp reaches only its lane quarter): each thread
    // decodes the 64 codes of its row and stores them as 32 columns of bf16 pairs.
    const int row = 32 * (warp & 3) + lane;
    const uint32_t tlane = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)S::kACol0;
    const int conv_n = u_end - u_begin;
    for (int g = 0; g < conv_n; ++g) {
      const int qs = g % NQ, as = g % NA;
      bool ok = mbar_wait(fullQ + 8 * qs, (g / NQ) & 1, abort_flag, pc.status);
      // the stage's previous tile has been multiplied (its MMAs' commit)
      ok = (g < NA || mbar_wait(emptyA + 8 * as, ((g / NA) - 1) & 1, abort_flag, pc.status)) && ok;
      tc_fence_after();
      if (__all_sync(0xffffffffu, ok)) {
        const uint4 *src = reinterpret_cast<const uint4 *>(qring + (size_t)qs * S::kQ + row * 32);
        const uint4 c0 = src[0], c1 = src[1];
        const uint32_t cw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
        uint32_t v[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint4 o = q4_to_bf16x8(cw[i]);
          v[4 * i] = o.x;
          v[4 * i + 1] = o.y;
          v[4 * i + 2] = o.z;
          v[4 * i + 3] = o.w;
        }
        tmem_st32(tlane + (uint32_t)(as * 32), v);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(emptyQ + 8 * qs);
        mbar_arrive(fullA + 8 * as);
      }
    }
    if (args.csplit) cluster_sync_all();
  } else {
    // ------------------------------------------------------------ drain + epilogues
    pdl_wait();  // norm sums, residuals and the outputs' earlier readers
    const int quad = warp & 3, chalf = warp >> 2, r = quad * 32 + lane;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const int nh_tiles = pc.n_embd / kTcK;
    int ch = 0;
    if constexpr (MODE == GM_LMHEAD) {
      if (tid < N) tb.run_best[tid] = 0ull;
    }
    uint32_t fix_phase = 0u;  // parity of fix_bar
    // per-item tables of the first item tile, while the first chunks are multiplied
    int tb_it = (int)(tc_seg(u_begin, u_end, ktiles).t % item_tiles);
    if (u_begin < u_end) tc_tables<N, MODE>(args, tb_it, tb);
    tc_epi_sync();
    float acc[H][NCH][16];
    bool cl_synced = false;  // cluster split-K: this thread passed the exchange barrier
    const uint32_t *szrow = nullptr;  // INT4: this thread's (scale, zero) row in the tile
    uint32_t szq[4] = {0u, 0u, 0u, 0u};  // INT4: its pairs of the next four groups
    int q4_g0 = 0, q4_g1 = 0;             // INT4: first and last group of the segment
    bool q4_staged = false;               // INT4: the segment's group sums are in qsum
    for (int u = u_begin; u < u_end;) {
      const TcSeg sg = tc_seg(u, u_end, ktiles);
      u += sg.kt1 - sg.kt0;
      if constexpr (Q4) {
        // INT4 applies the RMSNorm scales per group: the segment's item tables first
        const int it0 = sg.t % item_tiles;
        if (it0 != tb_it) {
          tc_epi_sync();
          tc_tables<N, MODE>(args, it0, tb);
          tc_epi_sync();
          tb_it = it0;
        }
        szrow = tc_q4_sz_row<MODE>(args, sg.t / item_tiles, r);
        // the groups this segment touches; their (scale, zero) pairs for this row four
        // groups ahead in registers, and the items' sums of x over them in shared memory
        // (read from global memory per chunk when they do not fit)
        q4_g0 = sg.kt0 >> 1;
        const int g1 = (sg.kt1 - 1) >> 1, ng = g1 - q4_g0 + 1;
        q4_g1 = g1;
#pragma unroll
        for (int d = 0; d < 4; ++d) szq[d] = (szrow && q4_g0 + d <= g1) ? __ldg(szrow + q4_g0 + d) : 0u;
        q4_staged = N * ng <= S::kQsumFloats;
        if (q4_staged) {
          const int GS = pc.K >> 7, i0 = it0 * N;
          tc_epi_sync();  // the previous segment's drains have read the buffer
          for (int idx = tid; idx < N * ng; idx += kTcEpiThreads) {
            const int gi = idx / N, c = idx - gi * N, item = i0 + c;
            qsum[idx] = item < args.M ? __ldcg(args.gsum + (size_t)item * GS + q4_g0 + gi) : 0.f;
          }
          tc_epi_sync();
        }
      }
#pragma unroll
      for (int h = 0; h < H; ++h)
#pragma unroll
        for (int j = 0; j < NCH; ++j)
#pragma unroll
          for (int i = 0; i < 16; ++i) acc[h][j][i] = 0.f;
      for (int cb = sg.kt0; cb < sg.kt1; ++ch) {
        const int ce = tc_chunk_end<H, CHK>(cb, sg.kt1, nh_tiles);
        const int h = tc_half<H>(cb, pc.n_embd);
        const int hb = ch % NBUF;
        if constexpr (Q4) {
          // chunks are whole 128-wide groups (or the part of one at a segment's edge), in
          // order: the group's scale for this row (queued four groups ahead), and the zero
          // point times each item's sum of x over the group for the chunk that holds the
          // group's first k-tile
          const int grp = cb >> 1;
          const bool first = (cb & 1) == 0;
          const uint32_t szv = szq[0];
          szq[0] = szq[1];
          szq[1] = szq[2];
          szq[2] = szq[3];
          szq[3] = (szrow && grp + 4 <= q4_g1) ? __ldg(szrow + grp + 4) : 0u;
          const float gs = bf_lo(szv), gz = first ? bf_hi(szv) : 0.f;
          const bool ok = mbar_wait(hi_full + 8 * hb, (ch / NBUF) & 1, abort_flag, pc.status);
          tc_fence_after();
          if (ok) {
#pragma unroll
            for (int j = 0; j < NCH; ++j) {
              if (!tc_has<N>(j, chalf)) continue;
              const uint32_t col = tmem + lane_base + S::buf_col(hb) + (uint32_t)tc_c0<N>(j, chalf);
              // x0, then x1 and x2 products, added in that order; then the group's affine
              // map and the item's RMSNorm scale
              float t[16], xs[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const int c = tc_c0<N>(j, chalf) + i;
                if (!first) {
                  xs[i] = 0.f;
                } else if (q4_staged) {
                  xs[i] = qsum[(grp - q4_g0) * N + c];
                } else {
                  const int item = (sg.t % item_tiles) * N + c;
                  xs[i] = item < args.M ? __ldcg(args.gsum + (size_t)item * (pc.K >> 7) + grp) : 0.f;
                }
              }
              {
                uint32_t raw[P][16];  // the parts' columns, loaded together, one wait
#pragma unroll
                for (int q = 0; q < P; ++q) tmem_ld16_async(col + (uint32_t)(q * N), raw[q]);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                  t[i] = __uint_as_float(raw[0][i]);
#pragma unroll
                  for (int q = 1; q < P; ++q) t[i] += __uint_as_float(raw[q][i]);
                }
              }
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const int c = tc_c0<N>(j, chalf) + i;
                const float ns = ModeTraits<MODE>::kNorm ? tb.scale[(c < N ? c : 0) * H + h] : 1.f;
                acc[0][j][i] = fmaf(ns, fmaf(gs, t[i], gz * xs[i]), acc[0][j][i]);
              }
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(hi_free + 8 * hb);
          cb = ce;
          continue;
        }
        const bool ok = mbar_wait(hi_full + 8 * hb, (ch / NBUF) & 1, abort_flag, pc.status);
        tc_fence_after();
        if (ok) {
          // x0, then x1 and x2 products of this chunk, added in that order
#pragma unroll
          for (int j = 0; j < NCH; ++j) {
            if (!tc_has<N>(j, chalf)) continue;
            const uint32_t col = tmem + lane_base + S::buf_col(hb) + (uint32_t)tc_c0<N>(j, chalf);
            uint32_t raw[P][16];  // the parts' columns, loaded together, one wait
#pragma unroll
            for (int q = 0; q < P; ++q) tmem_ld16_async(col + (uint32_t)(q * N), raw[q]);
            tmem_wait_ld();
            if (H == 2 && h == 1) {
#pragma unroll
              for (int q = 0; q < P; ++q)
#pragma unroll
                for (int i = 0; i < 16; ++i) acc[H - 1][j][i] += __uint_as_float(raw[q][i]);
            } else {
#pragma unroll
              for (int q = 0; q < P; ++q)
#pragma unroll
                for (int i = 0; i < 16; ++i) acc[0][j][i] += __uint_as_float(raw[q][i]);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(hi_free + 8 * hb);
        cb = ce;
      }
      const int rt = sg.t / item_tiles, it = sg.t % item_tiles;
      if (it != tb_it) {  // a tile of another item tile: its tables first
        tc_epi_sync();
        tc_tables<N, MODE>(args, it, tb);
        tc_epi_sync();
        tb_it = it;
      }
      // each K half's sum times its RMSNorm scale, the halves added: from here on a
      // tile's partial sums are one [N][128] block (INT4 applied the scales per group)
      if constexpr (Q4) {
      } else if constexpr (ModeTraits<MODE>::kNorm) {
#pragma unroll
        for (int j = 0; j < NCH; ++j)
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int c = tc_c0<N>(j, chalf) + i;
            float v = 0.f;
#pragma unroll
            for (int h = 0; h < H; ++h) v += acc[h][j][i] * tb.scale[(c < N ? c : 0) * H + h];
            acc[0][j][i] = v;
          }
      } else if constexpr (H == 2) {
#pragma unroll
        for (int j = 0; j < NCH; ++j)
#pragma unroll
          for (int i = 0; i < 16; ++i) acc[0][j][i] += acc[1][j][i];
      }
      unsigned ownm = ~0u;
      if (args.csplit) {
        // cluster split-K (one segment per CTA): this rank's partial tile into its idle
        // weight ring, one cluster barrier, then this rank's share of the columns summed
        // over the ranks in rank order, straight from their shared memory
        const int cs = args.csplit;
        const uint32_t rank = cluster_rank();
        float *red = reinterpret_cast<float *>(aring);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
#pragma unroll
        for (int j = 0; j < NCH; ++j)
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (tc_has<N>(j, chalf)) red[((size_t)tc_c0<N>(j, chalf) + i) * kTcM + r] = acc[0][j][i];
        cluster_sync_all();
        cl_synced = true;
        ownm = 0u;
#pragma unroll
        for (int j = 0; j < NCH; ++j) {
          const int cidx = N >= 32 ? 2 * j + chalf : 0;
          const bool mine = NCH >= cs ? (j % cs) == (int)rank : (cidx % cs) == (int)rank;
          if (mine && tc_has<N>(j, chalf)) ownm |= 1u << j;
        }
        const uint32_t red_addr = smem_addr(red);
#pragma unroll
        for (int j = 0; j < NCH; ++j) {
          if (!((ownm >> j) & 1u)) continue;
#pragma unroll
          for (int i = 0; i < 16; ++i) acc[0][j][i] = 0.f;
          const uint32_t off = (uint32_t)(((size_t)tc_c0<N>(j, chalf) * kTcM + r) * 4);
          for (int q = 0; q < cs; ++q) {
            const uint32_t src = dsmem_map(red_addr + off, (uint32_t)q);
            float v[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = ld_dsmem(src + (uint32_t)(i * kTcM * 4));
#pragma unroll
            for (int i = 0; i < 16; ++i) acc[0][j][i] += v[i];
          }
        }
      } else if (!(sg.kt0 == 0 && sg.kt1 == ktiles)) {
        // a shared tile: publish this CTA's raw sums; the last contributor adds them all
        const int t0 = sg.t * ktiles;
        const int c_first = sched.cta_of(t0), c_last = sched.cta_of(t0 + ktiles - 1);
        // slot 0: the CTA's first segment; slot 1: a later (its last) segment
        const int my_slot = sched.start(cta) >= t0 ? 0 : 1;
        // The CTA's last segment: when every other contributor has already arrived, this
        // CTA is the last and keeps its sums in registers (no publish, no arrival).
        bool last_known = false;
        if (u >= u_end) {
          if (tid == 0) {
            unsigned seen;
            asm volatile("ld.acquire.gpu.u32 %0, [%1];" : "=r"(seen) : "l"(args.tile_cnt + sg.t) : "memory");
            *last_sh = seen == (unsigned)(c_last - c_first) ? 1 : 0;
          }
          tc_epi_sync();
          last_known = *last_sh != 0;
        }
        if (!last_known) {
          float *mine = args.part + ((size_t)cta * 2 + my_slot) * N * kTcM;
#pragma unroll
          for (int j = 0; j < NCH; ++j)
#pragma unroll
            for (int i = 0; i < 16; ++i)
              if (tc_has<N>(j, chalf)) mine[((size_t)tc_c0<N>(j, chalf) + i) * kTcM + r] = acc[0][j][i];
          __threadfence();
          tc_epi_sync();
          if (tid == 0) {
            const unsigned prev = atomicAdd(args.tile_cnt + sg.t, 1u);
            *last_sh = prev == (unsigned)(c_last - c_first) ? 1 : 0;
          }
          tc_epi_sync();
          if (!*last_sh) continue;
        }
        __threadfence();
        // fixed order: the published sums of contributors c_first .. c_last (this CTA's
        // own included), one contributor's tile at a time
        auto part_of = [&](int cq) {  // a contributor's segment is its first (slot 0) unless it began earlier
          return args.part + ((size_t)cq * 2 + (sched.start(cq) >= t0 ? 0 : 1)) * N * kTcM;
        };
        if (u >= u_end) {
          // this CTA's last segment: its rings are idle, so one thread bulk-copies every
          // other contributor's published partial into them (all in flight at once), and
          // the rows are added in CTA order from shared memory; this CTA's own sums are
          // still in registers.
          constexpr int kPart = N * kTcM;  // floats per published partial
          constexpr int kCap = (int)(((size_t)NA * S::kAS + (size_t)NB * S::kBStage) / ((size_t)kPart * 4));
          static_assert(kCap >= 1, "a published partial fits the rings");
          const float *stg = reinterpret_cast<const float *>(aring);
          float own[NCH][16];
#pragma unroll
          for (int j = 0; j < NCH; ++j)
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              own[j][i] = acc[0][j][i];
              acc[0][j][i] = 0.f;
            }
          for (int c2 = c_first; c2 <= c_last; c2 += kCap) {
            const int cend = min(c_last, c2 + kCap - 1);
            const bool others = !(c2 == cend && c2 == cta);
            if (others) {
              if (tid == 0) {
                // the partials were written through the generic proxy by other CTAs and
                // acquired through the tile counter; order them before the bulk reads
                asm volatile("fence.proxy.async.global;" ::: "memory");
                mbar_expect_tx(fix_bar, (uint32_t)((cend - c2 + 1 - (cta >= c2 && cta <= cend ? 1 : 0)) * kPart * 4));
                const uint64_t pol = l2_evict_first_policy();
                for (int cq = c2; cq <= cend; ++cq)
                  if (cq != cta)
                    bulk_g2s(smem_addr(aring + (size_t)(cq - c2) * kPart * 4), part_of(cq), (uint32_t)(kPart * 4),
                             fix_bar, pol);
              }
              mbar_wait(fix_bar, fix_phase, abort_flag, pc.status);
              fix_phase ^= 1u;
            }
            for (int cq = c2; cq <= cend; ++cq) {
#pragma unroll
              for (int j = 0; j < NCH; ++j) {
                if (!tc_has<N>(j, chalf)) continue;
                if (cq == cta) {
#pragma unroll
                  for (int i = 0; i < 16; ++i) acc[0][j][i] += own[j][i];
                } else {
                  const float *src = stg + (size_t)(cq - c2) * kPart + (size_t)tc_c0<N>(j, chalf) * kTcM + r;
#pragma unroll
                  for (int i = 0; i < 16; ++i) acc[0][j][i] += src[(size_t)i * kTcM];
                }
              }
            }
            tc_epi_sync();  // every thread has read this batch before the next overwrites it
          }
        } else {
          // mid-share (the rings are still streaming this CTA's next tile): kU contributors
          // per pass, all their loads in flight together, added in CTA order
#pragma unroll
          for (int j = 0; j < NCH; ++j)
#pragma unroll
            for (int i = 0; i < 16; ++i) acc[0][j][i] = 0.f;
          constexpr int kVals = NCH * 16;
          constexpr int kU = kVals >= 64 ? 2 : (kVals >= 32 ? 4 : 8);
          for (int c2 = c_first; c2 <= c_last; c2 += kU) {
            const float *src[kU];
#pragma unroll
            for (int q = 0; q < kU; ++q) src[q] = part_of(min(c2 + q, c_last)) + r;  // past the last: not added
#pragma unroll
            for (int j = 0; j < NCH; ++j) {
              if (!tc_has<N>(j, chalf)) continue;
              float v[kU][16];
#pragma unroll
              for (int q = 0; q < kU; ++q)
#pragma unroll
                for (int i = 0; i < 16; ++i) v[q][i] = __ldcg(src[q] + ((size_t)tc_c0<N>(j, chalf) + i) * kTcM);
#pragma unroll
              for (int q = 0; q < kU; ++q)
                if (c2 + q <= c_last) {
#pragma unroll
                  for (int i = 0; i < 16; ++i) acc[0][j][i] += v[q][i];
                }
            }
          }
        }
        if (tid == 0) args.tile_cnt[sg.t] = 0u;
      }
      tc_tile_epilogue<N, MODE>(args, acc, rt, it, tb, ownm);
    }
    if (args.csplit && !cl_synced) cluster_sync_all();  // (a CTA without a segment)
    if constexpr (MODE == GM_LMHEAD) {
      // the last CTA to finish decodes every item's argmax
      if (args.item_tiles == 1) tc_lm_flush<N>(args, tb, 0);
      __threadfence();
      tc_epi_sync();
      if (tid == 0) {
        const unsigned prev = atomicAdd(pc.am_count, 1u);
        *last_sh = prev == gridDim.x - 1 ? 1 : 0;
      }
      tc_epi_sync();
      if (*last_sh) {
        __threadfence();
        lmhead_finalize(pc, 0, args.M, tid, kTcEpiThreads);
        if (tid == 0) *pc.am_count = 0u;
      }
    }
  }
  __syncthreads();
  // no CTA of a cluster leaves while a peer may still read its shared memory
  if (args.csplit) cluster_sync_all();
  if (warp == kTcMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(S::kTmemCols) : "memory");
  }
}

// ------------------------------------------------------------------ host side
// Tensor maps (gemm_tc.cu): bf16 rows with a (64 x box_rows) box and 128-byte swizzle;
// INT4 code rows with a (32-byte x box_rows) box.
bool tc_make_map(CUtensorMap *map, const void *base, int rows, int cols, int box_rows);
bool tc_make_code_map(CUtensorMap *map, const void *base, int rows, int K, int box_rows);

// Clusters of s CTAs (s = 2..8) of one instantiation that fit on the GPU at once (0: none,
// or not queried); filled by tc_prepare.
template <int N, int MODE, bool Q4>
struct TcClusterFit {
  static int n[9];
};
template <int N, int MODE, bool Q4>
int TcClusterFit<N, MODE, Q4>::n[9] = {};

// Cluster split-K width for `tiles` tiles of `ktiles` k-tiles: the s in 2..8 that keeps the
// most SMs busy (at least two k-tiles per rank, every cluster co-resident), used when it
// fills at least 60% of the SMs (any fill for TC_SCHED_CLUSTER); 0 = stream-K.  Measured
// on the drafter's batched projections, 96 of 152 SMs in clusters beat 152 in stream-K:
// the stream-K finisher's serial fix-up and epilogue cost more than the idle SMs.
inline int tc_pick_split(const int *fit, long long tiles, int ktiles, int num_sms, int policy) {
  if (policy == TC_SCHED_STREAM_K) return 0;
  int best = 0;
  long long best_ctas = 0;
  for (int cs = 2; cs <= 8; ++cs) {
    if (ktiles < 2 * cs || tiles * cs > num_sms) break;
    if (tiles > fit[cs]) continue;
    if (tiles * cs > best_ctas) {
      best = cs;
      best_ctas = tiles * cs;
    }
  }
  if (policy != TC_SCHED_CLUSTER && best_ctas * 5 < (long long)num_sms * 3) return 0;
  return best;
}

template <int N, int MODE, bool Q4>
static cudaError_t tc_launch_n(const TcLaunch &L, cudaStream_t st, bool pdl) {
  using S = TcShape<N, MODE, Q4>;
  TcArgs a;
  memset(&a, 0, sizeof(a));
  a.p = L.p;
  a.p.item0 = 0;
  a.p.items = L.M;
  a.M = L.M;
  a.sumsq = L.sumsq;
  a.part = L.part;
  a.tile_cnt = L.tile_cnt;
  const int K = L.p.K;
  if (K % kTcK || L.p.rows % (MODE == GM_GATEUP ? 128 : 1)) return cudaErrorInvalidValue;
  const int box_a = MODE == GM_GATEUP ? 64 : kTcM;
  if constexpr (Q4) {
    // INT4 codes, their (scale, zero) rows and the per-group sums of x
    if (K % 128 || !L.s0 || !L.gsum || L.sz_stride < K / 128) return cudaErrorInvalidValue;
    if (!tc_make_code_map(&a.a0, L.a0, L.a0_rows, K, box_a)) return cudaErrorInvalidValue;
    if (L.a1 && !tc_make_code_map(&a.a1, L.a1, L.a1_rows, K, box_a)) return cudaErrorInvalidValue;
    if (L.a2 && !tc_make_code_map(&a.a2, L.a2, L.a2_rows, K, box_a)) return cudaErrorInvalidValue;
    a.sz0 = L.s0;
    a.sz1 = L.s1;
    a.sz2 = L.s2;
    a.sz_stride = L.sz_stride;
    a.gsum = L.gsum;
  } else {
    if (!tc_make_map(&a.a0, L.a0, L.a0_rows, K, box_a)) return cudaErrorInvalidValue;
    if (L.a1 && !tc_make_map(&a.a1, L.a1, L.a1_rows, K, box_a)) return cudaErrorInvalidValue;
    if (L.a2 && !tc_make_map(&a.a2, L.a2, L.a2_rows, K, box_a)) return cudaErrorInvalidValue;
  }
  if (!tc_make_map(&a.b0, L.b0, L.M, K, N)) return cudaErrorInvalidValue;
  if (S::P > 1 && (!tc_make_map(&a.b1, L.b1, L.M, K, N) || !tc_make_map(&a.b2, L.b2, L.M, K, N)))
    return cudaErrorInvalidValue;
  a.row_tiles = (L.p.rows + kTcM - 1) / kTcM;
  a.item_tiles = (L.M + N - 1) / N;
  a.ktiles = K / kTcK;
  const long long tiles = (long long)a.row_tiles * a.item_tiles;
  const long long units = tiles * a.ktiles;
  if (units > (1ll << 30) || tiles > (long long)L.tile_cnt_elems) return cudaErrorInvalidValue;
  a.units = (int)units;
  a.csplit = tc_pick_split(TcClusterFit<N, MODE, Q4>::n, tiles, a.ktiles, L.num_sms, L.schedule);
  const int grid = a.csplit ? (int)tiles * a.csplit : (int)std::min<long long>(L.num_sms, units);
  // stream-K partials: two slots per CTA
  if (!a.csplit && (size_t)grid * 2 * N * kTcM > L.part_elems) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(Q4 ? kTcThreadsQ4 : kTcThreads);
  cfg.dynamicSmemBytes = S::kSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  if (a.csplit) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = (unsigned)a.csplit;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = (unsigned)na;
  return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<N, MODE, Q4>, a);
}

template <int MODE, bool Q4>
static cudaError_t tc_launch_mode(const TcLaunch &L, cudaStream_t st, bool pdl) {
  switch (tc_tile_items(L.M, MODE)) {
    case 16: return tc_launch_n<16, MODE, Q4>(L, st, pdl);
    case 32: return tc_launch_n<32, MODE, Q4>(L, st, pdl);
    case 64: return tc_launch_n<64, MODE, Q4>(L, st, pdl);
    default:
      if constexpr (TcMode<MODE>::kMaxN >= 128 && !Q4) return tc_launch_n<128, MODE, Q4>(L, st, pdl);
      return cudaErrorInvalidValue;
  }
}

template <int N, int MODE, bool Q4>
static cudaError_t tc_prepare_n() {
  cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<N, MODE, Q4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       TcShape<N, MODE, Q4>::kSmem);
  if (e != cudaSuccess) return e;
  for (int cs = 2; cs <= 8; ++cs) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cs);
    cfg.blockDim = dim3(Q4 ? kTcThreadsQ4 : kTcThreads);
    cfg.dynamicSmemBytes = TcShape<N, MODE, Q4>::kSmem;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = (unsigned)cs;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_tc_kernel<N, MODE, Q4>, &cfg) != cudaSuccess) {
      (void)cudaGetLastError();  // no cluster launches of this width: stream-K only
      n = 0;
    }
    TcClusterFit<N, MODE, Q4>::n[cs] = n;
  }
  return cudaSuccess;
}

template <int MODE, bool Q4>
static cudaError_t tc_prepare_mode() {
  cudaError_t e = tc_prepare_n<16, MODE, Q4>();
  if (e == cudaSuccess) e = tc_prepare_n<32, MODE, Q4>();
  if (e == cudaSuccess) e = tc_prepare_n<64, MODE, Q4>();
  if constexpr (TcMode<MODE>::kMaxN >= 128 && !Q4)
    if (e == cudaSuccess) e = tc_prepare_n<128, MODE, Q4>();
  return e;
}

}  // namespace e3
