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
// tiles (shallow ring: they come from L2).  Every mbarrier wait is bounded
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

// ------------------------------------------------------------------ shapes
template <int MODE>
struct TcMode {
  static constexpr int H = ModeTraits<MODE>::kHalves;
  static constexpr int P = MODE == GM_ENCODE ? 1 : 3;  // bf16 parts of x
  static constexpr int kMaxN = MODE == GM_ENCODE ? 128 : 64;
  static constexpr bool kStaging = MODE == GM_QKV || MODE == GM_GATEUP;  // row exchange
};

template <int N, int MODE>
struct TcShape {
  using T = TcMode<MODE>;
  static constexpr int H = T::H, P = T::P;
  static constexpr int kA = kTcM * kTcK * 2;            // 16 KB weight tile
  static constexpr int kB = N * kTcK * 2;               // one activation part
  static constexpr int kBStage = P * kB;
  // TMEM: two chunk buffers of [P][N] columns (a chunk lies in one K half)
  static constexpr int NP = P * N;                      // MMA width: the parts stacked
  static_assert(NP % 16 == 0 && NP <= 256, "MMA N of kind::f16 with M = 128");
  static constexpr int kCols = 2 * NP;
  static_assert(kCols <= 512, "accumulators fit in TMEM");
  static constexpr int kTmemCols = kCols <= 32 ? 32 : kCols <= 64 ? 64 : kCols <= 128 ? 128 : kCols <= 256 ? 256 : 512;
  static constexpr int NCH = N >= 32 ? N / 32 : 1;      // 16-column chunks per epilogue thread
  static constexpr int kStageBytes = T::kStaging ? kTcM * (N + 1) * 4 : 0;
  // lm_head: per-quad best keys of a tile [4][N] and the CTA's running best [N] (u64)
  static constexpr int kLmBytes = MODE == GM_LMHEAD ? 5 * N * 8 : 0;
  static constexpr int kAux = 3072;                      // barriers and per-item tables
  // activation ring: shallow (L2 hits); the weight ring (HBM) takes the rest
  static constexpr int kNB = kBStage <= 12 * 1024 ? 4 : 3;
  static constexpr int kFixed = 1024 /*alignment*/ + kAux + kStageBytes + kLmBytes + kNB * kBStage;
  static constexpr int kFitA = (int)((kTcSmemLimit - kFixed) / kA);
  static constexpr int kNA = kFitA > 12 ? 12 : kFitA;   // weight ring stages
  static_assert(kNA >= 4 && kNA >= kNB, "a weight ring of four stages, no shallower than the activation ring");
  static constexpr int kSmem = kFixed + kNA * kA;
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
template <int H>
__device__ __forceinline__ int tc_chunk_end(int cb, int kt1, int nh_tiles) {
  int ce = min(kt1, (cb / kTcChunk + 1) * kTcChunk);
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
template <int N, int MODE>
__global__ void __launch_bounds__(kTcThreads, 1) gemm_tc_kernel(const __grid_constant__ TcArgs args) {
  using S = TcShape<N, MODE>;
  constexpr int H = S::H, P = S::P, NA = S::kNA, NB = S::kNB, NCH = S::NCH;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  // [A ring NA x 16 KB][B ring NB x P parts][staging][barriers, flags, per-item tables]
  unsigned char *aring = smem;
  unsigned char *bring = aring + (size_t)NA * S::kA;
  float *stage = reinterpret_cast<float *>(bring + (size_t)NB * S::kBStage);
  unsigned char *lmb = reinterpret_cast<unsigned char *>(stage) + S::kStageBytes;
  unsigned char *aux = lmb + S::kLmBytes;
  const uint32_t fullA = smem_addr(aux), emptyA = fullA + 8 * NA;
  const uint32_t fullB = emptyA + 8 * NA;
  const uint32_t hi_full = fullB + 8 * NB, hi_free = hi_full + 16;
  const uint32_t mma_done = hi_free + 16;
  const uint32_t fix_bar = mma_done + 8;  // bulk copies of published partials (last tile)
  unsigned char *aux2 = aux + 8 * (2 * NA + 2 * NB + 7);
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
  static_assert(8 * (2 * S::kNA + 2 * S::kNB + 7) + 16 + 4 * (N * S::H + 4 * N) <= S::kAux, "aux area");

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
      mbar_init(fullA + 8 * i, 1);
      mbar_init(emptyA + 8 * i, 1);
    }
    for (int i = 0; i < NB; ++i) {
      mbar_init(fullB + 8 * i, 1);
    }
    for (int i = 0; i < 2; ++i) {
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
        __syncwarp();
      }
      u += sg.kt1 - sg.kt0;
    }
    for (int q = max(0, g - NA); q < g; ++q) tc_drain_wait(fullA + 8 * (q % NA), (q / NA) & 1);
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
        // slot s last held stage g - NB: free once that stage's MMAs finished, which the
        // weight ring's empty barrier of that stage records
        if (g >= NB && !warp_wait(emptyA + 8 * ((g - NB) % NA), ((g - NB) / NA) & 1, abort_flag, pc.status)) {
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
        const int ce = tc_chunk_end<H>(cb, sg.kt1, nh_tiles);
        const int hb = ch & 1;
        if (ch >= 2 && !warp_wait(hi_free + 8 * hb, ((ch >> 1) - 1) & 1, abort_flag, pc.status)) {
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
          const uint64_t ad0 = adesc0 + (uint64_t)((sa * S::kA) >> 4);
          const uint64_t bd0 = bdesc0 + (uint64_t)((sb * S::kBStage) >> 4);
          if (leader) {
#pragma unroll
            for (int kk = 0; kk < kTcK / 16; ++kk)  // 32 bytes further along K per slice
              tc_mma(dt, ad0 + (uint64_t)(kk * 2), bd0 + (uint64_t)(kk * 2), idesc, (kt > cb || kk > 0) ? 1u : 0u);
            tc_commit(emptyA + 8 * sa);  // both rings' slots are free once these MMAs finish
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
    for (int u = u_begin; u < u_end;) {
      const TcSeg sg = tc_seg(u, u_end, ktiles);
      u += sg.kt1 - sg.kt0;
#pragma unroll
      for (int h = 0; h < H; ++h)
#pragma unroll
        for (int j = 0; j < NCH; ++j)
#pragma unroll
          for (int i = 0; i < 16; ++i) acc[h][j][i] = 0.f;
      for (int cb = sg.kt0; cb < sg.kt1; ++ch) {
        const int ce = tc_chunk_end<H>(cb, sg.kt1, nh_tiles);
        const int h = tc_half<H>(cb, pc.n_embd);
        const int hb = ch & 1;
        const bool ok = mbar_wait(hi_full + 8 * hb, (ch >> 1) & 1, abort_flag, pc.status);
        tc_fence_after();
        if (ok) {
          // x0, then x1 and x2 products of this chunk, added in that order
#pragma unroll
          for (int j = 0; j < NCH; ++j) {
            if (!tc_has<N>(j, chalf)) continue;
            const uint32_t col = tmem + lane_base + S::buf_col(hb) + (uint32_t)tc_c0<N>(j, chalf);
#pragma unroll
            for (int q = 0; q < P; ++q) {
              if (H == 2 && h == 1) tmem_add16(col + (uint32_t)(q * N), acc[H - 1][j]);
              else tmem_add16(col + (uint32_t)(q * N), acc[0][j]);
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
      // tile's partial sums are one [N][128] block
      if constexpr (ModeTraits<MODE>::kNorm) {
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
          constexpr int kCap = (int)(((size_t)NA * S::kA + (size_t)NB * S::kBStage) / ((size_t)kPart * 4));
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
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D bf16 tensor map over a row-major [rows, cols] matrix with a (64 x box_rows) box and
// 128-byte swizzle.
bool tc_make_map(CUtensorMap *map, const void *base, int rows, int cols, int box_rows) {
  auto fn = encode_fn();
  if (!fn || !base || (reinterpret_cast<uintptr_t>(base) & 15u) || cols % 64 || rows < 1) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)kTcK, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Clusters of s CTAs (s = 2..8) of one instantiation that fit on the GPU at once (0: none,
// or not queried); filled by tc_prepare.
template <int N, int MODE>
struct TcClusterFit {
  static int n[9];
};
template <int N, int MODE>
int TcClusterFit<N, MODE>::n[9] = {};

// Cluster split-K width for `tiles` tiles of `ktiles` k-tiles: the s in 2..8 that keeps the
// most SMs busy (at least two k-tiles per rank, every cluster co-resident), used when it
// fills at least 60% of the SMs (any fill for TC_SCHED_CLUSTER); 0 = stream-K.  Measured
// on the drafter's batched projections, 96 of 152 SMs in clusters beat 152 in stream-K:
// the stream-K finisher's serial fix-up and epilogue cost more than the idle SMs.
static int tc_pick_split(const int *fit, long long tiles, int ktiles, int num_sms, int policy) {
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

template <int N, int MODE>
static cudaError_t tc_launch_n(const TcLaunch &L, cudaStream_t st, bool pdl) {
  using S = TcShape<N, MODE>;
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
  if (!tc_make_map(&a.a0, L.a0, L.a0_rows, K, box_a)) return cudaErrorInvalidValue;
  if (L.a1 && !tc_make_map(&a.a1, L.a1, L.a1_rows, K, box_a)) return cudaErrorInvalidValue;
  if (L.a2 && !tc_make_map(&a.a2, L.a2, L.a2_rows, K, box_a)) return cudaErrorInvalidValue;
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
  a.csplit = tc_pick_split(TcClusterFit<N, MODE>::n, tiles, a.ktiles, L.num_sms, L.schedule);
  const int grid = a.csplit ? (int)tiles * a.csplit : (int)std::min<long long>(L.num_sms, units);
  // stream-K partials: two slots per CTA
  if (!a.csplit && (size_t)grid * 2 * N * kTcM > L.part_elems) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kTcThreads);
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
  return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<N, MODE>, a);
}

// Items per tile: the smallest of 16, 32, 64 (128 for the one-part encode) that holds M;
// more items take several item tiles.
int tc_tile_items(int M, int mode) {
  const int cap = mode == GM_ENCODE ? TcMode<GM_ENCODE>::kMaxN : TcMode<GM_QKV>::kMaxN;
  int n = 16;
  while (n < M && n < cap) n *= 2;
  return n;
}

template <int MODE>
static cudaError_t tc_launch_mode(const TcLaunch &L, cudaStream_t st, bool pdl) {
  switch (tc_tile_items(L.M, MODE)) {
    case 16: return tc_launch_n<16, MODE>(L, st, pdl);
    case 32: return tc_launch_n<32, MODE>(L, st, pdl);
    case 64: return tc_launch_n<64, MODE>(L, st, pdl);
    default:
      if constexpr (TcMode<MODE>::kMaxN >= 128) return tc_launch_n<128, MODE>(L, st, pdl);
      return cudaErrorInvalidValue;
  }
}

cudaError_t tc_launch(const TcLaunch &L, cudaStream_t st, bool pdl) {
  switch (L.p.mode) {
    case GM_ENCODE: return tc_launch_mode<GM_ENCODE>(L, st, pdl);
    case GM_QKV: return tc_launch_mode<GM_QKV>(L, st, pdl);
    case GM_O: return tc_launch_mode<GM_O>(L, st, pdl);
    case GM_GATEUP: return tc_launch_mode<GM_GATEUP>(L, st, pdl);
    case GM_DOWN: return tc_launch_mode<GM_DOWN>(L, st, pdl);
    case GM_LMHEAD: return tc_launch_mode<GM_LMHEAD>(L, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}

template <int N, int MODE>
static cudaError_t tc_prepare_n() {
  cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<N, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       TcShape<N, MODE>::kSmem);
  if (e != cudaSuccess) return e;
  for (int cs = 2; cs <= 8; ++cs) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cs);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = TcShape<N, MODE>::kSmem;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = (unsigned)cs;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_tc_kernel<N, MODE>, &cfg) != cudaSuccess) {
      (void)cudaGetLastError();  // no cluster launches of this width: stream-K only
      n = 0;
    }
    TcClusterFit<N, MODE>::n[cs] = n;
  }
  return cudaSuccess;
}

template <int MODE>
static cudaError_t tc_prepare_mode() {
  cudaError_t e = tc_prepare_n<16, MODE>();
  if (e == cudaSuccess) e = tc_prepare_n<32, MODE>();
  if (e == cudaSuccess) e = tc_prepare_n<64, MODE>();
  if constexpr (TcMode<MODE>::kMaxN >= 128)
    if (e == cudaSuccess) e = tc_prepare_n<128, MODE>();
  return e;
}

cudaError_t tc_prepare() {
  if (!encode_fn()) return cudaErrorNotSupported;
  cudaError_t e = tc_prepare_mode<GM_ENCODE>();
  if (e == cudaSuccess) e = tc_prepare_mode<GM_QKV>();
  if (e == cudaSuccess) e = tc_prepare_mode<GM_O>();
  if (e == cudaSuccess) e = tc_prepare_mode<GM_GATEUP>();
  if (e == cudaSuccess) e = tc_prepare_mode<GM_DOWN>();
  if (e == cudaSuccess) e = tc_prepare_mode<GM_LMHEAD>();
  return e;
}

// ------------------------------------------------------------------ activation prep
constexpr int kPrepIters = 8;  // 8-element vectors per thread: K up to 8 * 256 * 8 = 16384
// x (times the norm gain where the op normalises) split into three bf16 parts
// x0 = bf16(x), x1 = bf16(x - x0), x2 = bf16(x - x0 - x1) -- both differences are exact
// in float32 and x0 + x1 + x2 carries x's 24 significant bits -- and the sum of squares
// per item and K half for the deferred RMSNorm scale.  One CTA per item.
template <int MODE>
__global__ void __launch_bounds__(256) tc_prep_kernel(const GemvParams p, uint16_t *x0, uint16_t *x1,
                                                      uint16_t *x2, float *sumsq) {
  using T = ModeTraits<MODE>;
  constexpr int H = T::kHalves;
  __shared__ float red[8][H];
  pdl_trigger();
  pdl_wait();
  const int item = blockIdx.x, tid = threadIdx.x;
  const int K = p.K, KV = K >> 3;
  float ss[H];
#pragma unroll
  for (int h = 0; h < H; ++h) ss[h] = 0.f;
  uint4 *d0 = reinterpret_cast<uint4 *>(x0 + (size_t)item * K);
  uint4 *d1 = reinterpret_cast<uint4 *>(x1 + (size_t)item * K);
  uint4 *d2 = reinterpret_cast<uint4 *>(x2 + (size_t)item * K);
  auto pack = [](const uint16_t (&u)[8]) {
    return make_uint4(u[0] | ((uint32_t)u[1] << 16), u[2] | ((uint32_t)u[3] << 16),
                      u[4] | ((uint32_t)u[5] << 16), u[6] | ((uint32_t)u[7] << 16));
  };
  auto put = [&](int kv, const float (&x)[8]) {
    uint16_t u0[8], u1[8], u2[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      u0[i] = f2bf(x[i]);
      const float r1 = x[i] - bf1(u0[i]);
      u1[i] = f2bf(r1);
      u2[i] = f2bf(r1 - bf1(u1[i]));
    }
    d0[kv] = pack(u0);
    d1[kv] = pack(u1);
    d2[kv] = pack(u2);
  };
  if constexpr (MODE == GM_QKV) {
    const int n = p.n_embd, NV = n >> 3;
    const PairItem itm = resolve_pair(p.pairs, item, n);
    int tok = itm.tok;
    if (tok < 0 || tok >= p.target_vocab) {
      if (tid == 0 && (itm.write_kv || p.row_base == 0)) set_status(p.status, EAGLE3_DEV_BAD_TOKEN);
      tok = 0;
    }
    const uint4 *er = reinterpret_cast<const uint4 *>(p.embed + (size_t)tok * n);
    const float4 *gr = reinterpret_cast<const float4 *>(itm.g);
    const uint4 *wi = reinterpret_cast<const uint4 *>(p.norm0);
    const uint4 *wh = reinterpret_cast<const uint4 *>(p.norm1);
    // every load of this thread first (all in flight together), then convert and store
    constexpr int kIt = kPrepIters / 2;
    uint4 ue[kIt], uw[kIt], uh[kIt];
    float4 ga[kIt], gb[kIt];
#pragma unroll
    for (int it = 0; it < kIt; ++it) {
      const int kv = tid + it * 256;
      if (kv < NV) {
        ue[it] = __ldg(er + kv);
        uw[it] = __ldg(wi + kv);
        uh[it] = __ldg(wh + kv);
        ga[it] = __ldcg(gr + 2 * kv);
        gb[it] = __ldcg(gr + 2 * kv + 1);
      }
    }
#pragma unroll
    for (int it = 0; it < kIt; ++it) {
      const int kv = tid + it * 256;
      if (kv >= NV) break;
      const uint4 u = ue[it], w = uw[it];
      const float e[8] = {bf_lo(u.x), bf_hi(u.x), bf_lo(u.y), bf_hi(u.y), bf_lo(u.z), bf_hi(u.z), bf_lo(u.w), bf_hi(u.w)};
      const float wf[8] = {bf_lo(w.x), bf_hi(w.x), bf_lo(w.y), bf_hi(w.y), bf_lo(w.z), bf_hi(w.z), bf_lo(w.w), bf_hi(w.w)};
      float x[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        ss[0] += e[i] * e[i];
        x[i] = e[i] * wf[i];
      }
      put(kv, x);
      const float4 a = ga[it], b = gb[it];
      const uint4 hw = uh[it];
      const float g[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
      const float hf[8] = {bf_lo(hw.x), bf_hi(hw.x), bf_lo(hw.y), bf_hi(hw.y), bf_lo(hw.z), bf_hi(hw.z), bf_lo(hw.w), bf_hi(hw.w)};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        ss[H - 1] += g[i] * g[i];
        x[i] = g[i] * hf[i];
      }
      put(NV + kv, x);
    }
  } else {
    const float4 *src = reinterpret_cast<const float4 *>(p.xf + (size_t)item * K);
    const uint4 *wn = reinterpret_cast<const uint4 *>(p.norm0);
    // every load of this thread first (all in flight together), then convert and store
    float4 va[kPrepIters], vb[kPrepIters];
    uint4 vw[kPrepIters];
#pragma unroll
    for (int it = 0; it < kPrepIters; ++it) {
      const int kv = tid + it * 256;
      if (kv < KV) {
        va[it] = __ldcg(src + 2 * kv);
        vb[it] = __ldcg(src + 2 * kv + 1);
        if constexpr (T::kNorm) vw[it] = __ldg(wn + kv);
      }
    }
#pragma unroll
    for (int it = 0; it < kPrepIters; ++it) {
      const int kv = tid + it * 256;
      if (kv >= KV) break;
      const float4 a = va[it], b = vb[it];
      float x[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
      if constexpr (T::kNorm) {
        const uint4 w = vw[it];
        const float wf[8] = {bf_lo(w.x), bf_hi(w.x), bf_lo(w.y), bf_hi(w.y), bf_lo(w.z), bf_hi(w.z), bf_lo(w.w), bf_hi(w.w)};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          ss[0] += x[i] * x[i];
          x[i] *= wf[i];
        }
      }
      put(kv, x);
    }
  }
  if constexpr (T::kNorm) {
#pragma unroll
    for (int h = 0; h < H; ++h) {
      float v = ss[h];
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if ((tid & 31) == 0) red[tid >> 5][h] = v;
    }
    __syncthreads();
    if (tid < H) {
      float t = 0.f;
      for (int w = 0; w < 8; ++w) t += red[w][tid];
      sumsq[(size_t)item * H + tid] = t;
    }
  }
}

cudaError_t tc_prep_launch(const GemvParams &p, int M, uint16_t *x0, uint16_t *x1, uint16_t *x2,
                           float *sumsq, cudaStream_t st, bool pdl) {
  if (p.K > kPrepIters * 256 * 8 || p.K % 8) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(M);
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  switch (p.mode) {
    case GM_QKV: return cudaLaunchKernelEx(&cfg, tc_prep_kernel<GM_QKV>, p, x0, x1, x2, sumsq);
    case GM_O: return cudaLaunchKernelEx(&cfg, tc_prep_kernel<GM_O>, p, x0, x1, x2, sumsq);
    case GM_GATEUP: return cudaLaunchKernelEx(&cfg, tc_prep_kernel<GM_GATEUP>, p, x0, x1, x2, sumsq);
    case GM_DOWN: return cudaLaunchKernelEx(&cfg, tc_prep_kernel<GM_DOWN>, p, x0, x1, x2, sumsq);
    case GM_LMHEAD: return cudaLaunchKernelEx(&cfg, tc_prep_kernel<GM_LMHEAD>, p, x0, x1, x2, sumsq);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace e3
