// qmv chain: a whole decode step of dependent fused packed linears (M = 1) in
// one persistent, cooperative launch.
//
// A decode step is a chain of matrix-vector products where each link reads
// (a slice of) an earlier link's output.  Launching them one by one costs a
// launch ramp and drain per link (the pages count ~678 dispatches per packed
// decode step: "epic: realize low-precision / quantized performance on the
// OpenXLA (IREE) backend", section "The measured fusion gate").  Here every CTA
// walks the same link list:
//   * its producer warp streams the CTA's row blocks of every link, in order,
//     into the shared-memory ring with bulk async copies.  Weights never
//     depend on earlier links, so streaming never waits on a dependency: while
//     the consumers wait for a link's input, the ring fills with that link's
//     (and later links') weights;
//   * its consumer warps, at the first block of a link, wait until every row
//     block of the input link has been published (a per-link completion
//     counter in global memory), stage that input as x, then consume the ring
//     exactly like the single-launch kernel (qmv_core.cuh);
//   * after its last row block of a link the CTA publishes them all: CTA
//     barrier, then one release add of its block count to the link's counter.
// All CTAs are co-resident (cooperative launch), links only wait on earlier
// links and every CTA processes its items in link order, so the waits always
// end; they are bounded anyway and report through a device status word.
//
// Scratch memory: one 32-bit completion counter per link, supplied by the
// caller (qlin_qmv_chain_workspace_size) and zeroed on the stream before the
// launch.

#include <algorithm>

#include "device_common.cuh"
#include "qlin_internal.h"
#include "qmv_core.cuh"
#include "sm100_ptx.cuh"

namespace qlin {

__device__ unsigned int g_chain_status = 0;

namespace {

using namespace qmvcore;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kProducerWarp = kConsumerWarps;
constexpr int kMaxLinks = 160;
constexpr int kR = 1;                       // rows per consumer warp per block
constexpr int kRB = kConsumerWarps * kR;    // rows per block

struct LinkDev {
  const uint32_t* wq;
  const void* scales;
  const void* biases;
  void* y;
  const void* x;  // this link's input (x0 or a slice of an earlier output)
  int N, K;
  int dep;        // link whose completion gates x, or -1
  int n_blocks;   // row blocks of kRB rows
  int n_kt;       // k-tiles per row
  int kt_bytes;   // bytes of a row per k-tile
  int cta_offset; // CTA that owns block 0 (spreads blocks of consecutive links)
  int scale_copy; // scales/biases bulk-copied with the weights
  int fast;       // 2048-code k-tiles with scales copied (qmv_core fast path)
};

struct ChainParams {
  LinkDev links[kMaxLinks];
  unsigned* counters;
  unsigned long long dep_wait_ns;  // limit of one wait for an input link
  int n_links;
  int stages;
  int stage_bytes;
  int rounds_max;    // x layout rounds of the longest K
  int stalled_link;  // tests only: readers of this link wait for one block too many (-1: none)
};

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// first block of link L owned by CTA c (>= n_blocks when it owns none)
__device__ __forceinline__ int first_block(const LinkDev& L, int c, int G) {
  return ((c - L.cta_offset) % G + G) % G;
}

template <int BITS, typename AT>
__global__ void __launch_bounds__(kThreads, 2) qmv_chain_kernel(const __grid_constant__ ChainParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  uint8_t* ring = smem;
  float* xs = reinterpret_cast<float*>(ring + size_t(p.stages) * p.stage_bytes);
  float2* xsum = reinterpret_cast<float2*>(xs + xs_floats(p.rounds_max, BITS));
  float2* sb32 = xsum + p.rounds_max * 32;  // [warp][kR][32] (fast path)
  uint64_t* bars = reinterpret_cast<uint64_t*>(sb32 + kConsumerWarps * kR * 32);
  const uint32_t ring_u32 = ptx::smem_u32(ring);
  const uint32_t full0 = ptx::smem_u32(bars), empty0 = full0 + 8u * p.stages;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int c = blockIdx.x, G = gridDim.x;

  if (tid == 0) {
    for (int s = 0; s < p.stages; ++s) {
      ptx::mbar_init(full0 + 8u * s, 1);
      ptx::mbar_init(empty0 + 8u * s, kConsumerWarps);
    }
    ptx::fence_mbar_init();
  }
  __syncthreads();

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    int u = 0, s = 0;
    uint32_t round = 0;
    bool ok = true;
    for (int l = 0; l < p.n_links && ok; ++l) {
      const LinkDev& L = p.links[l];
      const int row_bytes = L.K * BITS / 8;
      const int gpr = L.K / kGroup;
      const int kt_groups = L.kt_bytes * (8 / BITS) / kGroup;
      const uint32_t sb_bytes = L.scale_copy ? uint32_t(kt_groups * 2) : 0u;
      for (int j = first_block(L, c, G); j < L.n_blocks && ok; j += G) {
        const int row0 = j * kRB;
        const int nr = min(kRB, L.N - row0);
        for (int kt = 0; kt < L.n_kt; ++kt) {
          if (round > 0 && !ptx::mbar_wait(empty0 + 8u * s, (round - 1) & 1u)) {
            if (lane == 0) atomicOr(&g_chain_status, 1u);
            ok = false;
            break;
          }
          const uint32_t stage = ring_u32 + uint32_t(s) * uint32_t(p.stage_bytes);
          const uint32_t w_bytes = uint32_t(L.kt_bytes);
          if (lane == 0)
            ptx::mbar_arrive_expect_tx(full0 + 8u * s, uint32_t(nr) * (w_bytes + 2 * sb_bytes));
          __syncwarp();
          const uint8_t* wbase = reinterpret_cast<const uint8_t*>(L.wq);
          const AT* sc = static_cast<const AT*>(L.scales);
          const AT* bi = static_cast<const AT*>(L.biases);
          const uint32_t sb0 = stage + uint32_t(kRB) * w_bytes;
          if (L.n_kt == 1) {
            if (lane == 0) {
              bulk_copy(stage, wbase + int64_t(row0) * row_bytes, uint32_t(nr) * w_bytes,
                        full0 + 8u * s);
              if (L.scale_copy) {
                bulk_copy(sb0, sc + int64_t(row0) * gpr, uint32_t(nr) * sb_bytes, full0 + 8u * s);
                bulk_copy(sb0 + uint32_t(kRB) * sb_bytes, bi + int64_t(row0) * gpr,
                          uint32_t(nr) * sb_bytes, full0 + 8u * s);
              }
            }
          } else {
            for (int r = lane; r < nr; r += 32) {
              const int64_t row = row0 + r;
              bulk_copy(stage + uint32_t(r) * w_bytes,
                        wbase + row * row_bytes + int64_t(kt) * L.kt_bytes, w_bytes,
                        full0 + 8u * s);
              if (L.scale_copy) {
                const int64_t g0 = row * gpr + int64_t(kt) * kt_groups;
                bulk_copy(sb0 + uint32_t(r) * sb_bytes, sc + g0, sb_bytes, full0 + 8u * s);
                bulk_copy(sb0 + uint32_t(kRB + r) * sb_bytes, bi + g0, sb_bytes, full0 + 8u * s);
              }
            }
          }
          ++u;
          if (++s == p.stages) {
            s = 0;
            ++round;
          }
        }
      }
    }
    if (!ok) {
      const int first = u > p.stages ? u - p.stages : 0;
      for (int v = first; v < u; ++v)
        if (!ptx::mbar_wait(full0 + 8u * (v % p.stages), uint32_t(v / p.stages) & 1u))
          if (lane == 0) atomicOr(&g_chain_status, 16u);
    }
    return;
  }

  // --------------------------------------------------------------- consumers
  // Control flow here is the same on every consumer thread whatever happens:
  // a wait that gives up records the failure, so the named CTA barriers below
  // are always reached by all 256 threads (the results are then garbage and
  // the status word says so).  A dependency wait that gives up only skips the
  // later dependency waits: the ring waits go on, so every bulk copy the
  // producer issued has landed before the CTA exits.  A ring wait that gives
  // up skips the later ring waits (each would take the full limit).
  int s = 0;
  uint32_t round = 0;
  bool dep_ok = true, ring_ok = true;
  float2* sbw = sb32 + warp * kR * 32;
  for (int l = 0; l < p.n_links; ++l) {
    const LinkDev& L = p.links[l];
    const int j0 = first_block(L, c, G);
    if (j0 >= L.n_blocks) continue;  // this CTA owns no block of this link
    if (L.dep >= 0) {
      if (tid == 0 && dep_ok) {
        const unsigned target =
            unsigned(p.links[L.dep].n_blocks) + (L.dep == p.stalled_link ? 1u : 0u);
        const unsigned* ctr = p.counters + L.dep;
        if (ld_acquire(ctr) < target) {
          const uint64_t t0 = ptx::globaltimer_ns();
          for (uint32_t i = 1;; ++i) {
            if (ld_acquire(ctr) >= target) break;
            if ((i & 255u) == 0 && ptx::globaltimer_ns() - t0 > p.dep_wait_ns) {
              atomicOr(&g_chain_status, 4u);
              dep_ok = false;
              break;
            }
          }
        }
      }
      consumers_sync();
    }
    const int rounds = (L.K * BITS / 128 + 31) / 32;
    stage_x<BITS, 1, AT, true>(static_cast<const AT*>(L.x), L.K, 1, L.K, rounds, xs, xsum, tid);
    const int kt_groups = L.kt_bytes * (8 / BITS) / kGroup;
    const StageGeom geom{L.kt_bytes, kt_groups, rounds, L.K / kGroup, L.N};
    const AT* sc = static_cast<const AT*>(L.scales);
    const AT* bi = static_cast<const AT*>(L.biases);
    AT* y = static_cast<AT*>(L.y);
    for (int j = j0; j < L.n_blocks; j += G) {
      const int row0 = j * kRB + warp * kR;
      float2 acc[kR][1];
#pragma unroll
      for (int r = 0; r < kR; ++r) acc[r][0] = make_float2(0.0f, 0.0f);
      for (int kt = 0; kt < L.n_kt; ++kt) {
        if (ring_ok && !ptx::mbar_wait(full0 + 8u * s, round & 1u)) {
          if (lane == 0) atomicOr(&g_chain_status, 2u);
          ring_ok = false;
        }
        const uint8_t* stage = ring + size_t(s) * p.stage_bytes;
        if (L.fast) {
          stage_scales_f32<BITS, kR, AT>(stage, kRB, warp * kR, sbw, lane);
          accumulate_fixed<BITS, 1, kR, AT>(stage, warp * kR, kt, sbw, xs, 0, xsum, 0, lane, acc);
        } else {
          accumulate_stage<BITS, 1, kR, AT>(stage, kRB, warp * kR, kt, kt, geom, L.scale_copy != 0,
                                            sc, bi, row0, xs, xsum, lane, acc);
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(empty0 + 8u * s);
        if (++s == p.stages) {
          s = 0;
          ++round;
        }
      }
      store_rows<1, kR, AT>(acc, lane, row0, 0, L.N, 1, y, L.N);
    }
    // publish this CTA's blocks of the link at once: every consumer thread's
    // stores happen before the CTA barrier, and thread 0's release add at GPU
    // scope is ordered after the barrier (the pattern of a grid-wide barrier)
    consumers_sync();
    if (tid == 0) red_release_add(p.counters + l, unsigned((L.n_blocks - 1 - j0) / G + 1));
  }
}

// ------------------------------------------------------------------- host
template <int BITS, typename AT>
qlin_status launch_chain_t(const void* x0, const qlin_link* links, int n_links, void* ws,
                           const ChainWaitOptions& wo, cudaStream_t st) {
  auto kern = qmv_chain_kernel<BITS, AT>;
  ChainParams p;  // ~13 KB, passed by value as the kernel's parameter block
  p.n_links = n_links;
  p.counters = static_cast<unsigned*>(ws);
  p.dep_wait_ns = wo.dep_wait_ns;
  p.stalled_link = wo.stalled_link;
  int max_kt_bytes = 0, max_k = 0, max_groups = 0;
  for (int l = 0; l < n_links; ++l) {
    const qlin_link& in = links[l];
    LinkDev& L = p.links[l];
    L.wq = in.wq;
    L.scales = in.scales;
    L.biases = in.biases;
    L.y = in.y;
    L.N = int(in.N);
    L.K = int(in.K);
    L.dep = in.input;
    L.x = in.input < 0 ? x0
                       : static_cast<const void*>(static_cast<const uint8_t*>(links[in.input].y) +
                                                  int64_t(in.input_offset) * 2);
    L.n_blocks = (L.N + kRB - 1) / kRB;
    const int row_bytes = L.K * BITS / 8;
    const bool sb_aligned = reinterpret_cast<uintptr_t>(in.scales) % 16 == 0 &&
                            reinterpret_cast<uintptr_t>(in.biases) % 16 == 0;
    const int gpr = L.K / kGroup;
    L.fast = (L.K % FixedTile<BITS>::kCodes == 0 && sb_aligned) ? 1 : 0;
    if (L.fast) {
      L.kt_bytes = FixedTile<BITS>::kBytes;
      L.n_kt = row_bytes / L.kt_bytes;
    } else {
      int n_kt = 1;
      while (row_bytes / n_kt > 2048 || row_bytes % n_kt || (row_bytes / n_kt) % 16) ++n_kt;
      L.n_kt = n_kt;
      L.kt_bytes = row_bytes / n_kt;
    }
    const int kt_codes = L.kt_bytes * (8 / BITS);
    const int kt_groups = kt_codes / kGroup;
    L.scale_copy = kt_codes % kGroup == 0 && (kt_groups * 2) % 16 == 0 && (gpr * 2) % 16 == 0 &&
                   sb_aligned;
    max_kt_bytes = std::max(max_kt_bytes, L.kt_bytes);
    if (L.scale_copy) max_groups = std::max(max_groups, kt_groups);
    max_k = std::max(max_k, L.K);
  }
  p.stage_bytes = (kRB * max_kt_bytes + 4 * kRB * max_groups + 127) / 128 * 128;
  p.rounds_max = (max_k * BITS / 128 + 31) / 32;
  const size_t fixed = size_t(xs_floats(p.rounds_max, BITS)) * 4 + size_t(p.rounds_max) * 32 * 8 +
                       size_t(kConsumerWarps) * kR * 32 * 8;
  // ring of about 64 KB so that two CTAs share an SM
  p.stages = std::max(2, std::min(8, (64 * 1024) / p.stage_bytes));
  size_t smem = size_t(p.stages) * p.stage_bytes + fixed + size_t(p.stages) * 16;
  if (smem > 220 * 1024)
    return fail(QLIN_ERR_UNSUPPORTED, "qlin_qmv_chain: K=%d too large for the staged x", max_k);

  static int attr_dev = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (attr_dev != dev) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024) !=
        cudaSuccess)
      return check_launch("qlin_qmv_chain: cudaFuncSetAttribute");
    attr_dev = dev;
  }
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem) !=
          cudaSuccess ||
      per_sm < 1)
    return fail(QLIN_ERR_UNSUPPORTED, "qlin_qmv_chain: kernel does not fit on an SM");
  const int G = per_sm * sm_count();
  int cum = 0;
  for (int l = 0; l < n_links; ++l) {
    p.links[l].cta_offset = cum % G;
    cum += p.links[l].n_blocks;
  }
  cudaError_t e = cudaMemsetAsync(ws, 0, size_t(n_links) * sizeof(unsigned), st);
  if (e != cudaSuccess) return fail(QLIN_ERR_CUDA, "qlin_qmv_chain: %s", cudaGetErrorString(e));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(G), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(QLIN_ERR_CUDA, "qmv_chain_kernel launch: %s", cudaGetErrorString(e));
  }
  return check_launch("qmv_chain_kernel");
}

}  // namespace

int chain_max_links() { return kMaxLinks; }

qlin_status launch_qmv_chain(const void* x0, const qlin_link* links, int n_links, int bits,
                             qlin_dtype dtype, void* ws, const ChainWaitOptions& wo,
                             cudaStream_t st) {
  if (dtype == QLIN_F16)
    return bits == 4 ? launch_chain_t<4, __half>(x0, links, n_links, ws, wo, st)
                     : launch_chain_t<8, __half>(x0, links, n_links, ws, wo, st);
  return bits == 4 ? launch_chain_t<4, __nv_bfloat16>(x0, links, n_links, ws, wo, st)
                   : launch_chain_t<8, __nv_bfloat16>(x0, links, n_links, ws, wo, st);
}

cudaError_t chain_take_device_status(unsigned* flags) {
  unsigned v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_chain_status, sizeof(v));
  if (e != cudaSuccess) return e;
  const unsigned zero = 0;
  e = cudaMemcpyToSymbol(g_chain_status, &zero, sizeof(zero));
  *flags = v;
  return e;
}

}  // namespace qlin
