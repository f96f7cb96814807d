// Tensor-core (tcgen05) GEMM for the drafter's projections at batched sizes: the rows of
// a weight matrix against N activation rows (items) at once, so each weight byte is read
// from HBM once for the whole batch.
//
// y[item, row] = sum_k W[row, k] * x[item, k].  The MMA's M side is 128 weight rows, its N
// side the items (16..256), K in 64-element stages ("swap AB": the weights are the A
// operand, the activations the B operand; both K-major in shared memory, 128-byte
// swizzled, loaded by TMA).  float32 activations are split into three bf16 parts
// x = x0 + x1 + x2 (exact to float32's 24 bits) and every part is multiplied; bf16
// features (the encode) are one part.  The products of x0 rotate over up to four TMEM
// accumulators and those of x1 and x2 (2^-8 smaller) share one more, so that no float32
// accumulator takes more than a quarter of the K slices; the epilogue adds them in a
// fixed order.  Accumulators are read back with tcgen05.ld for the same fused epilogues
// as the CUDA-core GEMV (epilogue.cuh).  Matrices with few 128-row tiles split K across
// CTAs; the last CTA of a tile adds the splits in a fixed order.
//
// Warp roles (320 threads): warps 0-7 epilogue (two per TMEM lane quadrant), warp 8 TMA
// producer, warp 9 MMA issuer (one elected thread) and TMEM owner.  Every mbarrier wait
// is bounded (EAGLE3_DEV_TIMEOUT), and no copy is left in flight when the CTA finishes.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "epilogue.cuh"
#include "internal.h"

namespace e3 {

constexpr int kTcM = 128;          // MMA M (weight rows per tile)
constexpr int kTcK = 64;           // K per stage: one 128-byte swizzle row of bf16
constexpr int kTcThreads = 320;
constexpr int kTcProducerWarp = 8;
constexpr int kTcMmaWarp = 9;

struct TcArgs {
  CUtensorMap a0;   // weight matrix of the tile (q / fc / o / gate / down / lm_head)
  CUtensorMap a1;   // second matrix: k (q/k/v) or up (gate/up)
  CUtensorMap a2;   // third matrix: v (q/k/v)
  CUtensorMap b0;   // activations [M, K] bf16: the bf16 features, or x0 of the split
  CUtensorMap b1;   // x1 of the split
  CUtensorMap b2;   // x2 of the split
  GemvParams p;     // epilogue parameters; p.items / p.item0 set per item tile in-kernel
  const float *sumsq;  // [M][halves] sum of squares of the staged x (norm modes)
  float *part;         // split-K partials [ksplit][halves][item_tiles * N][rows]
  unsigned *tile_cnt;  // split-K arrival counters [row_tiles * item_tiles]
  int M;               // items in total
  int ksplit, kper;    // K splits and K columns per split (a multiple of 64)
  int item_tiles, row_tiles;
  int nstage;
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

// 16 consecutive float32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
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

// ------------------------------------------------------------------ row maps
// Logical row (relative to the tile) of physical A-tile row r: the tile's rows follow the
// weight matrix; the epilogues expect RoPE partners (i, i + R/2) and gate/up on adjacent
// logical rows.
template <int MODE>
__device__ __forceinline__ int tc_logical_row(const GemvParams &p, int lrow0, int r) {
  if constexpr (MODE == GM_GATEUP) {
    return r < 64 ? 2 * r : 2 * (r - 64) + 1;
  } else if constexpr (MODE == GM_QKV) {
    const int d = p.head_dim, R = p.rope_dims, half = R >> 1;
    const int qr = p.n_head * d, kr = p.n_head_kv * d;
    const int lr = p.row_base + lrow0 + r;  // physical == logical set within a tile
    if (lr >= qr + kr) return r;            // v rows are not rotated
    const int rr = lr < qr ? lr : lr - qr;
    const int hr = rr % d;
    if (hr >= R) return r;
    const int lh = hr < half ? 2 * hr : 2 * (hr - half) + 1;
    return r - hr + lh;
  } else {
    return r;
  }
}

// ------------------------------------------------------------------ kernel
template <int N, int MODE>
struct TcShape {
  static constexpr int H = ModeTraits<MODE>::kHalves;
  static constexpr int P = MODE == GM_ENCODE ? 1 : 3;  // bf16 parts of x
  static constexpr int kA = kTcM * kTcK * 2;            // 16 KB
  static constexpr int kB = N * kTcK * 2;               // per part
  static constexpr int kStage = kA + P * kB;
  static constexpr int kLo = P > 1 ? 1 : 0;             // accumulator of the x1, x2 products
  static constexpr int kFit = 512 / (H * N) - kLo;
  static constexpr int kAccHi = kFit > 4 ? 4 : (kFit < 1 ? 1 : kFit);  // rotating x0 accumulators
  static constexpr int kAcc = kAccHi + kLo;
  static constexpr int kCols = kAcc * H * N;
  static_assert(kCols <= 512, "accumulators fit in TMEM");
  static constexpr int kFitStages = (int)((kTcSmemLimit - 1024 - 64) / kStage);
  static constexpr int kNst = kFitStages > 8 ? 8 : kFitStages;  // ring stages
  static_assert(kNst >= 2, "two stages fit in shared memory");
  static_assert(kTcM * AccStride<N>::value * 4 <= kNst * kStage, "accumulator tile fits the ring");
  static constexpr int kTmemCols = kCols <= 32 ? 32 : kCols <= 64 ? 64 : kCols <= 128 ? 128 : kCols <= 256 ? 256 : 512;
  // TMEM column of accumulator a (0..kAccHi-1: x0 products; kAccHi: the rest) of half h
  static __device__ __forceinline__ uint32_t col(int a, int h) { return (uint32_t)((a * H + h) * N); }
};

template <int N, int MODE>
__global__ void __launch_bounds__(kTcThreads, 1) gemm_tc_kernel(const __grid_constant__ TcArgs args) {
  using S = TcShape<N, MODE>;
  constexpr int H = S::H;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // 1024-byte alignment for the swizzled tiles
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const int nst = args.nstage;
  const uint32_t full0 = smem_addr(smem + (size_t)nst * S::kStage);
  const uint32_t empty0 = full0 + 8 * nst;
  const uint32_t done_bar = empty0 + 8 * nst;
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + (size_t)nst * S::kStage + 16 * nst + 8);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + (size_t)nst * S::kStage + 16 * nst + 16);
  __shared__ float scale_sm[N * 2];
  __shared__ int last_sh;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const GemvParams &pc = args.p;
  // item tiles of one row tile are adjacent in launch order, so they share its weights in L2
  const int row_tiles = args.row_tiles;
  const int it = blockIdx.x % args.item_tiles;
  const int rt = (blockIdx.x / args.item_tiles) % row_tiles;
  const int ks = blockIdx.x / (args.item_tiles * row_tiles);
  const int lrow0 = rt * kTcM;                      // logical row of the tile (rel. row_base)
  const int item0 = it * N;
  const int k_begin = ks * args.kper;
  const int k_end = min(pc.K, k_begin + args.kper);
  const int n_stages = (k_end - k_begin + kTcK - 1) / kTcK;

  if (warp == kTcMmaWarp) {
    // TMEM for H accumulators of N columns
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_holder)),
                 "r"(S::kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 0) {
    for (int i = 0; i < nst; ++i) {
      mbar_init(full0 + 8 * i, 1);
      mbar_init(empty0 + 8 * i, 1);
    }
    mbar_init(done_bar, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  pdl_trigger();

  if (warp == kTcProducerWarp) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_map(&args.a0);
      tma_prefetch_map(&args.b0);
      const uint64_t pol_w = l2_evict_first_policy();
      uint64_t pol_x;
      asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol_x));
      // which matrix and physical rows hold this tile
      const CUtensorMap *amap = &args.a0;
      int arow = lrow0;
      if constexpr (MODE == GM_QKV) {
        const int qr = pc.n_head * pc.head_dim, kr = pc.n_head_kv * pc.head_dim;
        const int lr = pc.row_base + lrow0;
        if (lr < qr) {
          amap = &args.a0;
          arow = lr;
        } else if (lr < qr + kr) {
          amap = &args.a1;
          arow = lr - qr;
        } else {
          amap = &args.a2;
          arow = lr - qr - kr;
        }
      } else if constexpr (MODE == GM_GATEUP) {
        arow = lrow0 / 2;
      }
      bool waited = false;
      int issued = 0;
      for (int st = 0; st < n_stages; ++st) {
        const int slot = st % nst;
        if (st >= nst && !mbar_wait(empty0 + 8 * slot, ((st / nst) - 1) & 1, abort_flag, pc.status)) break;
        const int kx = k_begin + st * kTcK;
        const uint32_t sa = smem_addr(smem + (size_t)slot * S::kStage);
        const uint32_t sb = sa + S::kA;
        mbar_expect_tx(full0 + 8 * slot, (uint32_t)S::kStage);
        if constexpr (MODE == GM_GATEUP) {
          tma_load_2d(sa, &args.a0, kx, arow, full0 + 8 * slot, pol_w);
          tma_load_2d(sa + S::kA / 2, &args.a1, kx, arow, full0 + 8 * slot, pol_w);
        } else {
          tma_load_2d(sa, amap, kx, arow, full0 + 8 * slot, pol_w);
        }
        if (!waited) {  // the activations come from the previous kernel
          pdl_wait();
          waited = true;
        }
        tma_load_2d(sb, &args.b0, kx, item0, full0 + 8 * slot, pol_x);
        if constexpr (S::P > 1) {
          tma_load_2d(sb + S::kB, &args.b1, kx, item0, full0 + 8 * slot, pol_x);
          tma_load_2d(sb + 2 * S::kB, &args.b2, kx, item0, full0 + 8 * slot, pol_x);
        }
        issued = st + 1;
      }
      for (int st = max(0, issued - nst); st < issued; ++st)
        mbar_wait(full0 + 8 * (st % nst), (st / nst) & 1, abort_flag, pc.status);
      if (!waited) pdl_wait();
    }
  } else if (warp == kTcMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = tc_idesc(kTcM, N);
      const int nh = pc.n_embd;  // K of the first half (q/k/v: [embed ; g])
      uint32_t started = 0u;  // bit a * H + h: accumulator (a, h) holds a product
      int t = 0;              // K slice index within this split
      for (int st = 0; st < n_stages; ++st) {
        const int slot = st % nst;
        if (!mbar_wait(full0 + 8 * slot, (st / nst) & 1, abort_flag, pc.status)) break;
        tc_fence_after();
        const int kx = k_begin + st * kTcK;
        const int h = (H == 2 && kx >= nh) ? 1 : 0;
        const uint32_t sa = smem_addr(smem + (size_t)slot * S::kStage);
        const uint32_t sb = sa + S::kA;
        const int kcols = min(kTcK, k_end - kx);  // a multiple of 16 (K is a multiple of 64)
#pragma unroll
        for (int kk = 0; kk < kTcK / 16; ++kk, ++t) {
          if (kk * 16 >= kcols) break;
          const uint64_t ad = smem_desc_sw128(sa + kk * 32);
          const int a = t % S::kAccHi;
          const int bit = a * H + h;
          tc_mma(tmem + S::col(a, h), ad, smem_desc_sw128(sb + kk * 32), idesc, (started >> bit) & 1u);
          started |= 1u << bit;
          if constexpr (S::P > 1) {
            const int lb = S::kAccHi * H + h;
            tc_mma(tmem + S::col(S::kAccHi, h), ad, smem_desc_sw128(sb + S::kB + kk * 32), idesc,
                   (started >> lb) & 1u);
            started |= 1u << lb;
            tc_mma(tmem + S::col(S::kAccHi, h), ad, smem_desc_sw128(sb + 2 * S::kB + kk * 32), idesc, 1u);
          }
        }
        tc_commit(empty0 + 8 * slot);  // the stage's smem is free once these MMAs finish
      }
      tc_commit(done_bar);
    }
  } else {
    // ------------------------------------------------------------ epilogue warps
    pdl_wait();  // the norm sums and the outputs' other readers belong to earlier kernels
    const bool ok = mbar_wait(done_bar, 0, abort_flag, pc.status);
    tc_fence_after();
    // The K slices of a (split, half) pair come in runs of at least four consecutive
    // slices, so every accumulator of a half that this split touches received a product;
    // a half it does not touch is zero.
    bool has_h[H];
#pragma unroll
    for (int h = 0; h < H; ++h)
      has_h[h] = H == 1 ? (k_end > k_begin) : (h == 0 ? k_begin < pc.n_embd : k_end > pc.n_embd);
    const int quad = warp & 3, chalf = warp >> 2;
    const int r = quad * 32 + lane;  // physical row of the tile (TMEM lane)
    GemvParams p = pc;
    p.item0 = item0;
    p.items = min(N, args.M - item0);
    // RMSNorm scales of the tile's items (norm modes)
    if constexpr (ModeTraits<MODE>::kNorm) {
      for (int i = tid; i < N * H; i += kGemvThreads) {
        const int m = i / H, h = i % H;
        float s = 0.f;
        if (item0 + m < args.M) s = args.sumsq[(size_t)(item0 + m) * H + h];
        scale_sm[i] = rsqrtf(s / (float)(pc.K / H) + pc.eps);
      }
    }
    consumer_sync();
    constexpr int AS = AccStride<N>::value;
    float *accs = reinterpret_cast<float *>(smem);  // the ring is idle now: [128][AS]
    const int lr = tc_logical_row<MODE>(pc, lrow0, r);
    const int ncol = N / 2;  // columns per warp in the split-K reduction
    // TMEM is read in 16-column chunks; the two warps of a lane quadrant take alternate
    // chunks.  sum16 adds the accumulators of half h in a fixed order.
    auto sum16 = [&](int h, int c0, float (&y)[16]) {
#pragma unroll
      for (int i = 0; i < 16; ++i) y[i] = 0.f;
#pragma unroll
      for (int a = 0; a < S::kAcc; ++a) {
        float v[16];
        tmem_ld16(tmem + ((uint32_t)(quad * 32) << 16) + S::col(a, h) + (uint32_t)c0, v);
#pragma unroll
        for (int i = 0; i < 16; ++i) y[i] += v[i];
      }
    };
    if (args.ksplit == 1) {
      for (int c0 = chalf * 16; c0 < N; c0 += 32) {
        float y[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) y[i] = 0.f;
#pragma unroll
        for (int h = 0; h < H; ++h) {
          float v[16];
          sum16(h, c0, v);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float a = has_h[h] ? v[i] : 0.f;
            y[i] += ModeTraits<MODE>::kNorm ? a * scale_sm[(c0 + i) * H + h] : a;
          }
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) accs[(size_t)lr * AS + c0 + i] = ok ? y[i] : 0.f;
      }
    } else {
      // split K: publish this split's raw sums, the last split of the tile reduces
      const size_t rows_pad = (size_t)row_tiles * kTcM;
      const size_t cols_pad = (size_t)args.item_tiles * N;
      for (int c0 = chalf * 16; c0 < N; c0 += 32) {
#pragma unroll
        for (int h = 0; h < H; ++h) {
          float v[16];
          sum16(h, c0, v);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            args.part[(((size_t)ks * H + h) * cols_pad + item0 + c0 + i) * rows_pad + lrow0 + r] =
                (ok && has_h[h]) ? v[i] : 0.f;
        }
      }
      __threadfence();
      consumer_sync();
      if (tid == 0) {
        const unsigned prev = atomicAdd(args.tile_cnt + (size_t)it * row_tiles + rt, 1u);
        last_sh = (prev == (unsigned)args.ksplit - 1) ? 1 : 0;
      }
      consumer_sync();
      if (last_sh) {
        __threadfence();
        for (int c0 = chalf * ncol; c0 < (chalf + 1) * ncol; ++c0) {
          float y = 0.f;
#pragma unroll
          for (int h = 0; h < H; ++h) {
            float sum = 0.f;
            for (int q = 0; q < args.ksplit; ++q)
              sum += __ldcg(&args.part[(((size_t)q * H + h) * cols_pad + item0 + c0) * rows_pad + lrow0 + r]);
            y += ModeTraits<MODE>::kNorm ? sum * scale_sm[c0 * H + h] : sum;
          }
          accs[(size_t)lr * AS + c0] = y;
        }
        if (tid == 0) args.tile_cnt[(size_t)it * row_tiles + rt] = 0u;
      }
    }
    tc_fence_before();
    consumer_sync();
    if (args.ksplit == 1 || last_sh) {
      const int nrows = min(kTcM, pc.rows - lrow0);
      epilogue<N, MODE>(p, accs, lrow0, nrows);
    }
  }
  __syncthreads();
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

template <int N, int MODE>
static cudaError_t tc_launch_n(const TcLaunch &L, cudaStream_t st, bool pdl) {
  using S = TcShape<N, MODE>;
  TcArgs a;
  memset(&a, 0, sizeof(a));
  a.p = L.p;
  a.M = L.M;
  a.sumsq = L.sumsq;
  a.part = L.part;
  a.tile_cnt = L.tile_cnt;
  const int K = L.p.K;
  const int box_a = MODE == GM_GATEUP ? 64 : kTcM;
  if (!tc_make_map(&a.a0, L.a0, L.a0_rows, K, box_a)) return cudaErrorInvalidValue;
  if (L.a1 && !tc_make_map(&a.a1, L.a1, L.a1_rows, K, box_a)) return cudaErrorInvalidValue;
  if (L.a2 && !tc_make_map(&a.a2, L.a2, L.a2_rows, K, box_a)) return cudaErrorInvalidValue;
  if (!tc_make_map(&a.b0, L.b0, L.M, K, N)) return cudaErrorInvalidValue;
  if (S::P > 1 && (!tc_make_map(&a.b1, L.b1, L.M, K, N) || !tc_make_map(&a.b2, L.b2, L.M, K, N)))
    return cudaErrorInvalidValue;
  const int row_tiles = (L.p.rows + kTcM - 1) / kTcM;
  const int item_tiles = (L.M + N - 1) / N;
  // the lm_head's argmax counts one CTA per row tile of a single item tile
  if (MODE == GM_LMHEAD && item_tiles != 1) return cudaErrorInvalidValue;
  // split K until the grid covers the SMs (K ranges stay multiples of 64, >= 512 wide)
  int ksplit = 1;
  const int ktiles = K / kTcK;
  while (MODE != GM_LMHEAD && ksplit < 16 && row_tiles * item_tiles * (ksplit + 1) <= L.num_sms &&
         ktiles / (ksplit + 1) >= 8)
    ++ksplit;
  if (ksplit > 1 && (!L.part || (size_t)ksplit * S::H * row_tiles * kTcM * item_tiles * N > L.part_elems ||
                     (size_t)row_tiles * item_tiles > L.tile_cnt_elems))
    ksplit = 1;
  // equal K ranges of whole 64-column tiles; no split is left empty
  const int tiles_per = (ktiles + ksplit - 1) / ksplit;
  ksplit = (ktiles + tiles_per - 1) / tiles_per;
  a.ksplit = ksplit;
  a.kper = tiles_per * kTcK;
  a.item_tiles = item_tiles;
  a.row_tiles = row_tiles;
  const size_t base = (size_t)S::kStage;
  const int nst = S::kNst;
  a.nstage = nst;
  const size_t smem = 1024 + (size_t)nst * base + 16 * nst + 32;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(item_tiles * row_tiles * ksplit);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<N, MODE>, a);
}

template <int MODE>
static cudaError_t tc_launch_mode(const TcLaunch &L, cudaStream_t st, bool pdl) {
  switch (tc_tile_items(L.M, MODE)) {
    case 16: return tc_launch_n<16, MODE>(L, st, pdl);
    case 32: return tc_launch_n<32, MODE>(L, st, pdl);
    case 64: return tc_launch_n<64, MODE>(L, st, pdl);
    case 128: return tc_launch_n<128, MODE>(L, st, pdl);
    default:
      if constexpr (MODE == GM_ENCODE) return tc_launch_n<256, MODE>(L, st, pdl);
      return cudaErrorInvalidValue;
  }
}

// Items per tile: the smallest of 16..128 that holds M; the encode (one bf16 part, so a
// smaller stage) goes up to 256.
int tc_tile_items(int M, int mode) {
  if (M <= 16) return 16;
  if (M <= 32) return 32;
  if (M <= 64) return 64;
  if (M <= 128 || mode != GM_ENCODE) return 128;
  return 256;
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
  return cudaFuncSetAttribute(gemm_tc_kernel<N, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)kTcSmemLimit);
}

template <int MODE>
static cudaError_t tc_prepare_mode() {
  cudaError_t e = tc_prepare_n<16, MODE>();
  if (e == cudaSuccess) e = tc_prepare_n<32, MODE>();
  if (e == cudaSuccess) e = tc_prepare_n<64, MODE>();
  if (e == cudaSuccess) e = tc_prepare_n<128, MODE>();
  if constexpr (MODE == GM_ENCODE)
    if (e == cudaSuccess) e = tc_prepare_n<256, MODE>();
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
    for (int kv = tid; kv < NV; kv += 256) {
      const uint4 u = er[kv], w = wi[kv];
      const float e[8] = {bf_lo(u.x), bf_hi(u.x), bf_lo(u.y), bf_hi(u.y), bf_lo(u.z), bf_hi(u.z), bf_lo(u.w), bf_hi(u.w)};
      const float wf[8] = {bf_lo(w.x), bf_hi(w.x), bf_lo(w.y), bf_hi(w.y), bf_lo(w.z), bf_hi(w.z), bf_lo(w.w), bf_hi(w.w)};
      float x[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        ss[0] += e[i] * e[i];
        x[i] = e[i] * wf[i];
      }
      put(kv, x);
      const float4 a = gr[2 * kv], b = gr[2 * kv + 1];
      const uint4 hw = wh[kv];
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
    for (int kv = tid; kv < KV; kv += 256) {
      const float4 a = src[2 * kv], b = src[2 * kv + 1];
      float x[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
      if constexpr (T::kNorm) {
        const uint4 w = wn[kv];
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
