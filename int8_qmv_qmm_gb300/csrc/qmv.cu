// qmv: fused dequantise-into-matvec on CUDA cores for decode (small M).
//
// y[m][n] = sum_k x[m][k] * (q[n][k]*scale[n][g(k)] + bias[n][g(k)])
//
// The packed payload is streamed from HBM exactly once per M-tile and consumed
// straight out of shared memory: the reconstructed weight never exists outside
// registers ("track(upstream-iree): fused dequant->matmul for the packed int8
// bandwidth win", section "The blocker (measured)": materialising it is what
// made the unfused path slower than f16).  Any N >= 1 works, including N not a
// multiple of 4 ("Metal backend: import qmv_impl from MLX").
//
// Data movement.  A CTA owns row blocks of RB = 8*R consecutive rows
// (persistent: block b, b + grid, ...).  A block is cut into k-tiles of KT
// bytes per row; one (block, k-tile) is one pipeline stage.  A producer warp
// fills a ring of shared-memory stages with 1-D bulk async copies (one per
// row, so no register holds in-flight data and each CTA keeps S stages --
// 50-100 KB -- in flight), and, when scales/biases are 16-byte aligned per
// row slice, bulk-copies their slices too (otherwise the consumers read them
// from global memory).  Eight consumer warps compute.  The producer starts
// before the kernel waits for its predecessor on the stream, so with
// programmatic dependent launch the weights stream while the previous kernel
// finishes.
//
// The per-chunk arithmetic, the lane-transposed x layout and the butterfly
// reduction are in qmv_core.cuh.  Warp w computes rows w*R .. w*R+R-1 of each
// stage; lanes take consecutive 16-byte chunks.  For one token on 2048-code
// k-tiles with eight-row blocks, warp w instead takes rows 2(w%4), 2(w%4)+1
// over half w/4 of every tile ("K halves"): each x value a lane loads from
// shared memory then serves two rows, and the two warps of a row pair add
// their sums through shared memory (3.4% off the decode step).  No global
// workspace.
//
// Split of K.  When the row blocks are few and long (small N, long K), a
// thread-block cluster of 2, 4 or 8 CTAs shares each row block: CTA c takes
// an equal share of the row's k-tiles and stages only the part of x they
// read, and CTAs 1.. add their row sums into CTA 0's shared memory, which
// stores the rows (the "split-K where N is small" of the M = 1 path).
//
// Every mbarrier wait is bounded; a wait that gives up sets a device status
// bit and the CTA unwinds after its outstanding copies have landed.

#include <algorithm>
#include <cstdlib>

#include "device_common.cuh"
#include "qlin_internal.h"
#include "qmv_core.cuh"
#include "sm100_ptx.cuh"

namespace qlin {

__device__ unsigned int g_qmv_status = 0;

namespace {

using namespace qmvcore;
constexpr int kThreads = (kConsumerWarps + 1) * 32;  // + one producer warp
constexpr int kProducerWarp = kConsumerWarps;

struct Shape {
  int M, N, K;
  int C;            // 16-byte chunks per row
  int rounds;       // rounds of the lane-transposed x layout of one CTA's
                    // k range: ceil(C / split / 32)
  int kt_bytes;     // bytes of one row per k-tile (multiple of 16, divides the row)
  int n_kt;         // k-tiles per row
  int n_blocks;     // row blocks
  int split;        // CTAs per row block (a cluster; 1: no split of K)
  int kt_per_cta;   // k-tiles each CTA of a row block takes
  int stages;       // ring depth
  int stage_bytes;  // bytes of one stage (weights, then scales and biases)
  unsigned flags;
  Epilogue ep;      // layer bias and f32 output (qlin_linear_ex)
};

// MODE 0: generic k-tiles, scales read from global memory; 1: generic k-tiles,
// scales copied into the stage; 2: fixed 2048-code k-tiles with scales copied
// (the fast path); 3: as 2, for one token (MT = 1) and 8-row blocks, each warp
// taking R rows (2 or 4) over one R-th part of every k-tile (of the rounds of
// its lanes), so that every x value a lane loads serves R rows; the R warps of
// a row group add their sums through shared memory.  EPI: a linear layer's epilogue (bias,
// float32 output) is applied; a separate instance, so the plain path's code is
// untouched.
template <int BITS, int MT, int R, typename AT, int MODE, bool EPI>
__global__ void __launch_bounds__(kThreads, 2) qmv_kernel(
    const AT* __restrict__ x, const uint32_t* __restrict__ wq, const AT* __restrict__ scales,
    const AT* __restrict__ biases, AT* __restrict__ y, const Shape sh) {
  constexpr bool kScaleCopy = MODE != 0;
  constexpr bool kKH = MODE == 3;
  static_assert(!kKH || (MT == 1 && (R == 2 || R == 4) &&
                         FixedTile<BITS>::kRounds % R == 0),
                "K parts: one token, R rows per warp over R parts of whole rounds");
  constexpr int kRB = kKH ? kConsumerWarps : kConsumerWarps * R;
  // (K parts) row groups of R rows, each shared by R warps
  constexpr int kGroups = kKH ? kConsumerWarps / R : 1;
  extern __shared__ __align__(16) uint8_t smem[];
  const int K = sh.K, N = sh.N;
  const int row_bytes = K * BITS / 8;
  const int gpr = K / kGroup;
  const int kt_groups = sh.kt_bytes * (8 / BITS) / kGroup;  // groups per row per k-tile
  const int xs_m = xs_floats(sh.rounds, BITS);  // floats per row of x (transposed layout)

  // shared memory: [stages][stage_bytes] | x (f32) | xsum (f32x2) | scale pairs | barriers
  //                | split-K receive buffer [split-1][warp][R*MT] (f32)
  uint8_t* ring = smem;
  float* xs = reinterpret_cast<float*>(ring + size_t(sh.stages) * sh.stage_bytes);
  float2* xsum = reinterpret_cast<float2*>(xs + MT * xs_m);
  float2* sb32 = xsum + MT * sh.rounds * 32;  // [warp][R][32] (fast path)
  uint64_t* bars = reinterpret_cast<uint64_t*>(sb32 + kConsumerWarps * R * 32);
  const uint32_t ring_u32 = ptx::smem_u32(ring);
  const uint32_t full0 = ptx::smem_u32(bars), empty0 = full0 + 8u * sh.stages;
  float* red = reinterpret_cast<float*>(bars + 2 * sh.stages);
  // (K parts) [2 buffers][row groups][R-1 parts][R rows] partial sums (at
  // most 48 floats), then a flag a consumer sets when one of its waits gave up
  float* kh_red = red;
  volatile int* kh_abort = reinterpret_cast<volatile int*>(red + 48);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int m0 = blockIdx.y * MT;
  // split > 1: a cluster of `split` CTAs shares one row block, CTA c taking
  // k-tiles [c, c+1) * kt_per_cta; otherwise the grid is persistent over the
  // row blocks
  const int split = sh.split;
  const int crank = split > 1 ? int(ptx::cluster_ctarank()) : 0;
  const int blk0 = split > 1 ? int(blockIdx.x) / split : int(blockIdx.x);
  const int blk_step = split > 1 ? sh.n_blocks : int(gridDim.x);
  const int kt_lo = crank * sh.kt_per_cta, kt_hi = kt_lo + sh.kt_per_cta;

  // the next kernel may launch at once: it only streams its own (read-only)
  // weights before its own dependency wait, which this kernel's completion
  // releases (0.3% faster on the decode step than triggering after the wait)
  grid_launch_dependents();
  if (tid == 0) {
    for (int s = 0; s < sh.stages; ++s) {
      ptx::mbar_init(full0 + 8u * s, 1);
      ptx::mbar_init(empty0 + 8u * s, kConsumerWarps);
    }
    if constexpr (kKH) *kh_abort = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  // (split-K) first half of the barrier that tells every CTA of the cluster
  // that the others have started: their shared memory may then be written
  if (split > 1) ptx::cluster_arrive_relaxed();

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    // stage s is filled for the (round+1)-th time after the consumers released
    // it round times: wait for completion number round-1 of its empty barrier
    int s = 0, issued = 0;
    uint32_t round = 0;
    bool ok = true;
    const uint32_t w_bytes = uint32_t(sh.kt_bytes);
    const uint32_t sb_bytes = kScaleCopy ? uint32_t(kt_groups * 2) : 0u;
    for (int blk = blk0; blk < sh.n_blocks && ok; blk += blk_step) {
      const int row0 = blk * kRB;
      const int nr = min(kRB, N - row0);
      for (int kt = kt_lo; kt < kt_hi; ++kt) {
        if (round > 0 && !ptx::mbar_wait(empty0 + 8u * s, (round - 1) & 1u)) {
          if (lane == 0) atomicOr(&g_qmv_status, 1u);
          ok = false;
          break;
        }
        const uint32_t stage = ring_u32 + uint32_t(s) * uint32_t(sh.stage_bytes);
        const uint32_t sb0 = stage + uint32_t(kRB) * w_bytes;
        if (lane == 0)
          ptx::mbar_arrive_expect_tx(full0 + 8u * s, uint32_t(nr) * (w_bytes + 2 * sb_bytes));
        __syncwarp();
        if (sh.n_kt == 1) {
          // whole rows: the block is one contiguous range (and so are its
          // scales and biases)
          if (lane == 0) {
            bulk_copy(stage, reinterpret_cast<const uint8_t*>(wq) + int64_t(row0) * row_bytes,
                      uint32_t(nr) * w_bytes, full0 + 8u * s);
            if constexpr (kScaleCopy) {
              const int64_t g0 = int64_t(row0) * gpr;
              bulk_copy(sb0, scales + g0, uint32_t(nr) * sb_bytes, full0 + 8u * s);
              bulk_copy(sb0 + uint32_t(kRB) * sb_bytes, biases + g0, uint32_t(nr) * sb_bytes,
                        full0 + 8u * s);
            }
          }
        } else {
          for (int r = lane; r < nr; r += 32) {
            const int64_t row = row0 + r;
            bulk_copy(stage + uint32_t(r) * w_bytes,
                      reinterpret_cast<const uint8_t*>(wq) + row * row_bytes +
                          int64_t(kt) * sh.kt_bytes,
                      w_bytes, full0 + 8u * s);
            if constexpr (kScaleCopy) {
              const int64_t g0 = row * gpr + int64_t(kt) * kt_groups;
              bulk_copy(sb0 + uint32_t(r) * sb_bytes, scales + g0, sb_bytes, full0 + 8u * s);
              bulk_copy(sb0 + uint32_t(kRB + r) * sb_bytes, biases + g0, sb_bytes,
                        full0 + 8u * s);
            }
          }
        }
        ++issued;
        if (++s == sh.stages) {
          s = 0;
          ++round;
        }
      }
    }
    if (!ok) {
      // let the copies already issued land before the CTA's memory goes away
      const int first = issued > sh.stages ? issued - sh.stages : 0;
      for (int v = first; v < issued; ++v)
        if (!ptx::mbar_wait(full0 + 8u * (v % sh.stages), uint32_t(v / sh.stages) & 1u))
          if (lane == 0) atomicOr(&g_qmv_status, 16u);
    }
    if (split > 1) {
      // the producer takes part in the cluster barriers of the reduction
      __syncwarp();
      ptx::cluster_wait();
      ptx::cluster_arrive_release();
      ptx::cluster_wait();
    }
    return;
  }

  // --------------------------------------------------------------- consumers
  // x is produced by the preceding kernel: wait for it (a no-op unless this is
  // a programmatic dependent launch).
  grid_dependency_wait();
  // a split CTA stages only the part of x its k-tiles read
  const int k_lo = kt_lo * sh.kt_bytes * (8 / BITS);
  stage_x<BITS, MT, AT, false>(x + int64_t(m0) * K + k_lo, K, sh.M - m0,
                               sh.kt_per_cta * sh.kt_bytes * (8 / BITS), sh.rounds, xs, xsum, tid);

  const StageGeom geom{sh.kt_bytes, kt_groups, sh.rounds, gpr, N};
  float2* sbw = sb32 + warp * R * 32;
  // this warp's first row within a block, and (K parts) its row group and
  // its part of the tile
  const int kh_group = kKH ? warp % kGroups : 0;
  const int w_row0 = kKH ? R * kh_group : warp * R;
  const int khalf = kKH ? warp / kGroups : 0;
  int s = 0, kh_buf = 0;
  uint32_t round = 0;
  for (int blk = blk0; blk < sh.n_blocks; blk += blk_step) {
    const int rb0 = blk * kRB + w_row0;  // this warp's first row
    float2 acc[R][MT];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int mm = 0; mm < MT; ++mm) acc[r][mm] = make_float2(0.0f, 0.0f);
    bool failed = false;
    for (int kt = kt_lo; kt < kt_hi; ++kt) {
      if constexpr (kKH) {
        // the warps of a row pair meet at a named barrier after every block:
        // a warp whose wait gave up carries on without computing (and tells
        // the others to stop waiting), so that its partner is never left
        // waiting at that barrier
        if (*kh_abort || !ptx::mbar_wait(full0 + 8u * s, round & 1u)) {
          if (lane == 0 && !*kh_abort) {
            atomicOr(&g_qmv_status, 2u);
            *kh_abort = 1;
          }
          __syncwarp();
          failed = true;
          if (++s == sh.stages) {
            s = 0;
            ++round;
          }
          continue;
        }
      } else if (!ptx::mbar_wait(full0 + 8u * s, round & 1u)) {
        if (lane == 0) atomicOr(&g_qmv_status, 2u);
        // no CTA-wide barrier follows: leaving is safe, except that a split
        // CTA still takes part in the cluster barriers below
        if (split == 1) return;
        failed = true;
        break;
      }
      const uint8_t* stage = ring + size_t(s) * sh.stage_bytes;
      if constexpr (kKH) {
        constexpr int kPartRounds = FixedTile<BITS>::kRounds / R;
        stage_scales_f32<BITS, R, AT>(stage, kRB, w_row0, sbw, lane);
        // (the part index selects compile-time round ranges)
        if (khalf == 0)
          accumulate_fixed<BITS, MT, R, AT, 0, kPartRounds>(stage, w_row0, kt - kt_lo, sbw, xs,
                                                            xs_m, xsum, sh.rounds * 32, lane,
                                                            acc);
        else if (khalf == 1)
          accumulate_fixed<BITS, MT, R, AT, kPartRounds, kPartRounds>(
              stage, w_row0, kt - kt_lo, sbw, xs, xs_m, xsum, sh.rounds * 32, lane, acc);
        else if constexpr (R == 4) {
          if (khalf == 2)
            accumulate_fixed<BITS, MT, R, AT, 2 * kPartRounds, kPartRounds>(
                stage, w_row0, kt - kt_lo, sbw, xs, xs_m, xsum, sh.rounds * 32, lane, acc);
          else
            accumulate_fixed<BITS, MT, R, AT, 3 * kPartRounds, kPartRounds>(
                stage, w_row0, kt - kt_lo, sbw, xs, xs_m, xsum, sh.rounds * 32, lane, acc);
        }
      } else if constexpr (MODE == 2) {
        stage_scales_f32<BITS, R, AT>(stage, kRB, warp * R, sbw, lane);
        accumulate_fixed<BITS, MT, R, AT>(stage, warp * R, kt - kt_lo, sbw, xs, xs_m, xsum,
                                          sh.rounds * 32, lane, acc);
      } else {
        accumulate_stage<BITS, MT, R, AT>(stage, kRB, warp * R, kt, kt - kt_lo, geom, kScaleCopy,
                                          scales, biases, rb0, xs, xsum, lane, acc);
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(empty0 + 8u * s);
      if (++s == sh.stages) {
        s = 0;
        ++round;
      }
    }
    const AT* lbias = EPI ? static_cast<const AT*>(sh.ep.bias) : nullptr;
    const bool yf32 = EPI && sh.ep.y_f32 != 0;
    if constexpr (kKH) {
      // the warps of parts 1.. of a row group hand their row sums to the
      // part-0 warp, which adds them to its own in part order and stores the
      // rows; two buffers by block parity, so a warp a block ahead never
      // overwrites sums not yet read
      using RS = RowSums<MT, R>;
      float total = RS::reduce(acc, lane);
      const int vi = RS::value_index(lane);
      float* pr = kh_red + (kh_buf * kGroups + kh_group) * (R - 1) * R;
      if (khalf > 0 && RS::owner(lane)) pr[(khalf - 1) * R + vi] = total;
      asm volatile("bar.sync %0, %1;" ::"r"(3 + kh_group), "n"(32 * R) : "memory");
      if (khalf == 0) {
        for (int p = 0; p < R - 1; ++p) total += pr[p * R + vi];
        const int row = rb0 + vi;
        if (RS::owner(lane) && row < N && !failed && !*kh_abort)
          store_value<AT>(total, row, m0, static_cast<void*>(y), N, lbias, yf32);
      }
      kh_buf ^= 1;
      continue;
    }
    if (split == 1) {
      store_rows<MT, R, AT>(acc, lane, rb0, m0, N, sh.M, static_cast<void*>(y), N, lbias, yf32);
      continue;
    }
    // ------------------------------------------------ split-K reduction
    // Every CTA reduces its partial sums across lanes; CTAs 1.. store theirs
    // into CTA 0's receive buffer, and CTA 0 adds them in rank order to its
    // own and stores the rows.  (With split > 1 this loop runs once.)
    using RS = RowSums<MT, R>;
    float total = RS::reduce(acc, lane);
    const int vi = RS::value_index(lane);
    ptx::cluster_wait();  // every CTA of the cluster has started
    if (crank != 0 && RS::owner(lane) && !failed)
      ptx::st_cluster_f32(
          ptx::map_shared_rank(ptx::smem_u32(red + ((crank - 1) * kConsumerWarps + warp) * RS::kV +
                                             vi),
                               0u),
          total);
    ptx::cluster_arrive_release();
    ptx::cluster_wait();  // the partials are in CTA 0's buffer
    if (crank == 0) {
      for (int src = 0; src < split - 1; ++src)
        total += red[(src * kConsumerWarps + warp) * RS::kV + vi];
      const int row = rb0 + vi / MT, m = m0 + vi % MT;
      if (RS::owner(lane) && row < N && m < sh.M)
        store_value<AT>(total, row, m, static_cast<void*>(y), N, lbias, yf32);
    }
  }
}

// ------------------------------------------------------------------- host
size_t smem_for(const Shape& sh, int MT, int R, int bits) {
  const int cw = 128 / bits;
  // ... + the split-K receive buffer, or 16 partial sums and a flag (K halves)
  return size_t(sh.stages) * sh.stage_bytes + size_t(MT) * sh.rounds * 32 * cw * 4 +
         size_t(MT) * sh.rounds * 32 * 8 + size_t(kConsumerWarps) * R * 32 * 8 +
         size_t(sh.stages) * 16 + size_t(sh.split - 1) * kConsumerWarps * R * MT * 4 + 208;
}

template <int BITS, int MT, int R, typename AT, int MODE, bool EPI>
qlin_status launch_t(const void* x, const uint32_t* wq, const void* scales, const void* biases,
                     void* y, const Shape& sh, size_t smem, cudaStream_t st) {
  auto kern = qmv_kernel<BITS, MT, R, AT, MODE, EPI>;
  // per device: attribute set once; occupancy cached per dynamic smem size
  static int attr_dev = -1;
  static size_t occ_smem[8] = {0};
  static int occ_blocks[8] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (attr_dev != dev) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024) !=
        cudaSuccess)
      return check_launch("qmv: cudaFuncSetAttribute");
    for (int i = 0; i < 8; ++i) occ_smem[i] = 0;
    attr_dev = dev;
  }
  int blocks_per_sm = 0;
  for (int i = 0; i < 8 && !blocks_per_sm; ++i)
    if (occ_smem[i] == smem) blocks_per_sm = occ_blocks[i];
  if (!blocks_per_sm) {
    int b = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kern, kThreads, smem) != cudaSuccess ||
        b < 1)
      b = 1;
    blocks_per_sm = b;
    int slot = 0;
    while (slot < 7 && occ_smem[slot]) ++slot;
    occ_smem[slot] = smem;
    occ_blocks[slot] = b;
  }
  // QLIN_QMV_CTAS_PER_SM caps the persistent grid below the occupancy limit,
  // leaving room on each SM for the next launch's CTAs (tuning)
  if (const char* env = std::getenv("QLIN_QMV_CTAS_PER_SM")) {
    const int v = std::atoi(env);
    if (v >= 1 && v < blocks_per_sm) blocks_per_sm = v;
  }
  const int64_t m_tiles = (sh.M + MT - 1) / MT;
  if (m_tiles > 65535) return fail(QLIN_ERR_UNSUPPORTED, "qlin_qmv: M too large");
  const int64_t resident = int64_t(blocks_per_sm) * sm_count();
  const int64_t per_tile = std::max<int64_t>(1, resident / std::min<int64_t>(m_tiles, resident));
  // split K: exactly one cluster of `split` CTAs per row block (the kernel's
  // reduction relies on it); otherwise persistent over the row blocks
  const int64_t gx = sh.split > 1
                         ? int64_t(sh.n_blocks) * sh.split
                         : std::max<int64_t>(1, std::min<int64_t>(sh.n_blocks, per_tile));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(gx), unsigned(m_tiles), 1u);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  unsigned n_attr = 0;
  if (sh.flags & QLIN_OVERLAP_PREVIOUS) {
    attr[n_attr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n_attr].val.programmaticStreamSerializationAllowed = 1;
    ++n_attr;
  }
  if (sh.split > 1) {
    attr[n_attr].id = cudaLaunchAttributeClusterDimension;
    attr[n_attr].val.clusterDim.x = unsigned(sh.split);
    attr[n_attr].val.clusterDim.y = 1;
    attr[n_attr].val.clusterDim.z = 1;
    ++n_attr;
  }
  cfg.attrs = n_attr ? attr : nullptr;
  cfg.numAttrs = n_attr;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, static_cast<const AT*>(x), wq,
                                           static_cast<const AT*>(scales),
                                           static_cast<const AT*>(biases), static_cast<AT*>(y),
                                           sh);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(QLIN_ERR_CUDA, "qmv_kernel launch: %s", cudaGetErrorString(e));
  }
  return check_launch("qmv_kernel");
}

// Rows per consumer warp: two (x reuse, fewer blocks) when rows are
// plentiful, one when the launch would otherwise leave SMs idle (four rows
// per warp needs ~150 registers and halves the resident warps: slower).
// QLIN_QMV_R (1 or 2) overrides it, for tuning.
int rows_per_warp(int64_t N, int64_t sms) {
  if (const char* env = std::getenv("QLIN_QMV_R")) {
    const int v = std::atoi(env);
    if (v == 1 || v == 2) return v;
  }
  return N >= 16 * 2 * sms ? 2 : 1;
}

// CTAs per row block.  K is split over a cluster only when the row blocks are
// too few to occupy the SMs (two CTAs each) and long: a split costs about
// 1 us (cluster launch and barriers) whatever its size, which a block of up
// to 16 KB of packed weights does not win back (measured on 300 x 512,
// 512 x 2048 and 1029 x 2048), while 129 rows of K = 8192 at 4 bits (32 KB a
// block) fell from 6.0 to 4.1 us.  The factor is the largest of 8, 4, 2 whose
// CTAs fit at once and leave each CTA at least 4 KB of the block.
// QLIN_QMV_SPLIT (1, 2, 4 or 8) overrides the choice, for tuning, wherever
// each CTA's share of a row is still a whole number of 16-byte chunks.
constexpr int64_t kMinSplitBlockBytes = 32 * 1024;
constexpr int64_t kMinSplitShareBytes = 4 * 1024;

int qmv_split(int n_blocks, int row_bytes, int rows_per_block, int sms) {
  auto divides = [&](int s) { return row_bytes % (16 * s) == 0; };
  if (const char* env = std::getenv("QLIN_QMV_SPLIT")) {
    const int v = std::atoi(env);
    if (v == 1 || v == 2 || v == 4 || v == 8) return divides(v) ? v : 1;
  }
  const int64_t block_bytes = int64_t(rows_per_block) * row_bytes;
  if (block_bytes < kMinSplitBlockBytes) return 1;
  for (int s = 8; s >= 2; s /= 2)
    if (int64_t(n_blocks) * s <= 2 * int64_t(sms) && divides(s) &&
        block_bytes / s >= kMinSplitShareBytes)
      return s;
  return 1;
}

template <int BITS, int MT, typename AT>
qlin_status dispatch_mt(const void* x, const uint32_t* wq, const void* scales,
                        const void* biases, void* y, Shape sh, cudaStream_t st) {
  const int64_t sms = sm_count();
  const int row_bytes = sh.K * BITS / 8;
  const int gpr = sh.K / kGroup;
  const int R = rows_per_warp(sh.N, sms);
  const int RB = kConsumerWarps * R;
  const bool sb_aligned = (reinterpret_cast<uintptr_t>(scales) % 16) == 0 &&
                          (reinterpret_cast<uintptr_t>(biases) % 16) == 0;
  const int n_blocks = (sh.N + RB - 1) / RB;
  const int split = qmv_split(n_blocks, row_bytes, RB, int(sms));
  sh.split = split;
  int mode;
  if (sh.K % (FixedTile<BITS>::kCodes * split) == 0 && sb_aligned) {
    // fast path: 2048-code k-tiles, scales copied into the stage
    mode = 2;
    sh.kt_bytes = FixedTile<BITS>::kBytes;
    sh.n_kt = row_bytes / sh.kt_bytes;
  } else {
    // k-tile: stages of about 32 KB of weights: the whole row (or the CTA's
    // share of it) when it fits, else the smallest split into equal
    // 16-byte-multiple tiles that does; a multiple of `split` tiles
    const int kt_max = std::max(512, 32768 / RB);
    int n_kt = split;
    while (row_bytes / n_kt > kt_max || row_bytes % n_kt || (row_bytes / n_kt) % 16) n_kt += split;
    sh.n_kt = n_kt;
    sh.kt_bytes = row_bytes / n_kt;
    const int kt_codes = sh.kt_bytes * (8 / BITS);
    const int kt_groups = kt_codes / kGroup;
    mode = (kt_codes % kGroup == 0 && (kt_groups * 2) % 16 == 0 && (gpr * 2) % 16 == 0 &&
            sb_aligned)
               ? 1
               : 0;
  }
  const int kt_groups = sh.kt_bytes * (8 / BITS) / kGroup;
  sh.stage_bytes = RB * sh.kt_bytes + (mode != 0 ? 2 * RB * kt_groups * 2 : 0);
  sh.stage_bytes = (sh.stage_bytes + 127) / 128 * 128;
  sh.n_blocks = n_blocks;
  sh.kt_per_cta = sh.n_kt / split;
  sh.rounds = (sh.C / split + 31) / 32;
  // ring depth: about 96 KB of stages, so that two CTAs fit on an SM
  // (QLIN_QMV_RING_KB overrides the target, for tuning)
  int ring_kb = 96;
  if (const char* env = std::getenv("QLIN_QMV_RING_KB")) {
    const int v = std::atoi(env);
    if (v >= 16 && v <= 200) ring_kb = v;
  }
  // one token on fixed k-tiles with one row per warp: the K-parts layout
  // (mode 3: R rows per warp, each over an R-th of every tile) instead, with
  // R = 2 (decode step: 358 us against 370 without; R = 4, possible where a
  // tile has 4 rounds, measured 367).  QLIN_QMV_KH (0, 2 or 4) overrides it,
  // for tuning.
  int kh = (MT == 1 && mode == 2 && R == 1 && split == 1) ? 2 : 0;
  if (const char* env = std::getenv("QLIN_QMV_KH")) {
    const int v = std::atoi(env);
    if (v == 0 || v == 2 || (v == 4 && FixedTile<BITS>::kRounds % 4 == 0)) kh = kh ? v : 0;
  }
  const int r_smem = kh ? kh : R;  // rows per warp that size the scale pairs
  sh.stages = std::max(2, std::min(8, (ring_kb * 1024) / sh.stage_bytes));
  size_t smem = smem_for(sh, MT, r_smem, BITS);
  while (sh.stages > 2 && smem > 110 * 1024) {
    --sh.stages;
    smem = smem_for(sh, MT, r_smem, BITS);
  }
  if (smem > 220 * 1024)
    return fail(QLIN_ERR_UNSUPPORTED, "qlin_qmv: K=%d too large for the staged x", sh.K);
  const bool epi = sh.ep.bias != nullptr || sh.ep.y_f32;
  if constexpr (MT == 1) {
    if constexpr (FixedTile<BITS>::kRounds % 4 == 0) {
      if (kh == 4)
        return epi ? launch_t<BITS, 1, 4, AT, 3, true>(x, wq, scales, biases, y, sh, smem, st)
                   : launch_t<BITS, 1, 4, AT, 3, false>(x, wq, scales, biases, y, sh, smem, st);
    }
    if (kh == 2)
      return epi ? launch_t<BITS, 1, 2, AT, 3, true>(x, wq, scales, biases, y, sh, smem, st)
                 : launch_t<BITS, 1, 2, AT, 3, false>(x, wq, scales, biases, y, sh, smem, st);
  }
#define QLIN_QMV_LAUNCH(RR, E)                                                                  \
  return mode == 2   ? launch_t<BITS, MT, RR, AT, 2, E>(x, wq, scales, biases, y, sh, smem, st)  \
         : mode == 1 ? launch_t<BITS, MT, RR, AT, 1, E>(x, wq, scales, biases, y, sh, smem, st)  \
                     : launch_t<BITS, MT, RR, AT, 0, E>(x, wq, scales, biases, y, sh, smem, st)
  if (epi) {
    if (R == 2) QLIN_QMV_LAUNCH(2, true);
    QLIN_QMV_LAUNCH(1, true);
  }
  if (R == 2) QLIN_QMV_LAUNCH(2, false);
  QLIN_QMV_LAUNCH(1, false);
#undef QLIN_QMV_LAUNCH
}

template <int BITS, typename AT>
qlin_status dispatch(const void* x, const uint32_t* wq, const void* scales, const void* biases,
                     void* y, int64_t M, int64_t N, int64_t K, unsigned flags,
                     const Epilogue& ep, cudaStream_t st) {
  Shape sh{};
  sh.flags = flags;
  sh.ep = ep;
  sh.M = int(M);
  sh.N = int(N);
  sh.K = int(K);
  sh.C = int(K * BITS / 128);
  sh.rounds = (sh.C + 31) / 32;
  const int MT = M >= 3 ? 4 : int(M);
  switch (MT) {
    case 1: return dispatch_mt<BITS, 1, AT>(x, wq, scales, biases, y, sh, st);
    case 2: return dispatch_mt<BITS, 2, AT>(x, wq, scales, biases, y, sh, st);
    default: return dispatch_mt<BITS, 4, AT>(x, wq, scales, biases, y, sh, st);
  }
}

}  // namespace

qlin_status launch_qmv(const void* x, const uint32_t* wq, const void* scales, const void* biases,
                       void* y, int64_t M, int64_t N, int64_t K, int bits, qlin_dtype dtype,
                       unsigned flags, const Epilogue& ep, cudaStream_t st) {
  if (dtype == QLIN_F16)
    return bits == 4 ? dispatch<4, __half>(x, wq, scales, biases, y, M, N, K, flags, ep, st)
                     : dispatch<8, __half>(x, wq, scales, biases, y, M, N, K, flags, ep, st);
  return bits == 4 ? dispatch<4, __nv_bfloat16>(x, wq, scales, biases, y, M, N, K, flags, ep, st)
                   : dispatch<8, __nv_bfloat16>(x, wq, scales, biases, y, M, N, K, flags, ep,
                                                st);
}

int qmv_plan_split(int64_t N, int64_t K, int bits, int sms) {
  const int RB = kConsumerWarps * rows_per_warp(N, sms);
  return qmv_split(int((N + RB - 1) / RB), int(K * bits / 8), RB, sms);
}

cudaError_t qmv_take_device_status(unsigned* flags) {
  unsigned v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_qmv_status, sizeof(v));
  if (e != cudaSuccess) return e;
  const unsigned zero = 0;
  e = cudaMemcpyToSymbol(g_qmv_status, &zero, sizeof(zero));
  *flags = v;
  return e;
}

}  // namespace qlin
